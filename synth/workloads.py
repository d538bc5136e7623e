"""The five synthetic workloads of the ZeRO++ codec path: shapes and input recipes.

Pure data: sizes, topologies, block sizes, bit widths, Adam hyper-parameters
and the ``synth.Recipe`` of every input tensor.  No codec arithmetic.

Input recipe (every workload): bf16 weights N(0, 0.02) from stream
``WEIGHTS`` indexed by global parameter index; the fp32 Adam master is the
exact widening of those weights; m = v = 0 and step t = 1 unless a test says
otherwise; rank r's gradient bucket comes from stream ``grad_stream(r)``
indexed by position in the bucket; a standalone Adam shard of n parameters
has gradients N(0, 1e-3) from stream ``SHARD_GRAD`` and its master widened
from the weights at global indices [bucket, bucket + n).
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import Dist, Recipe

WEIGHT_RECIPE = Recipe(Dist("normal", 0.02))
GRAD_NORMAL = Recipe(Dist("normal", 1e-3))
# two-hop bucket: Student-t (3 dof) x 1e-3, 0.1% of 256-element blocks carry
# one element scaled x100
GRAD_T3_OUTLIERS = Recipe(Dist("student_t", 1e-3, 3.0), outlier_block=256,
                          outlier_prob=1e-3, outlier_factor=100.0)
MOMENT_M_RECIPE = Recipe(Dist("normal", 1e-4))
MOMENT_V_RECIPE = Recipe(Dist("halfnormal", 1e-6))


@dataclass(frozen=True)
class Adam:
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    step: int = 1


@dataclass(frozen=True)
class QwZ:
    """qwZ on the weights: ``nranks`` shards of ``shard`` elements per call,
    ``calls`` calls (a long model streamed in chunks), the last call's shard
    replaced by ``tail_shard`` when nonzero."""
    nranks: int
    shard: int
    block: int
    bits: int = 8
    calls: int = 1
    tail_shard: int = 0

    @property
    def phi(self) -> int:
        if self.tail_shard:
            return self.nranks * (self.shard * (self.calls - 1) + self.tail_shard)
        return self.nranks * self.shard * self.calls


@dataclass(frozen=True)
class QgZ:
    nodes: int
    gpus_per_node: int
    bucket: int
    block: int
    bits: int = 4
    grad: Recipe = GRAD_NORMAL

    @property
    def nd(self) -> int:
        return self.nodes * self.gpus_per_node

    @property
    def slice_elems(self) -> int:
        return self.bucket // self.nd


@dataclass(frozen=True)
class Workload:
    name: str
    qwz: QwZ | None
    qgz: QgZ | None
    fused_adam: bool = True          # Adam fused onto the final hop
    standalone_adam: int = 0         # extra standalone Adam over this many params
    adam: Adam = field(default_factory=Adam)
    seed: int = 0


TINY = Workload(
    "tiny: Phi=2^20, N_d=4 (2x2), qwZ int8 B=256, qgZ int4 B=256",
    qwz=QwZ(nranks=4, shard=1 << 18, block=256, bits=8),
    qgz=QgZ(nodes=2, gpus_per_node=2, bucket=1 << 20, block=256, bits=4),
)

LLAMA_PHI = 4096 * 4096 * 4 + 4096 * 11008 * 3          # 202,375,168
LLAMA = Workload(
    "llama-layer bucket: Phi=202,375,168, N_d=8 (1x8), qwZ int8 B=512, qgZ int4 B=512",
    qwz=QwZ(nranks=8, shard=LLAMA_PHI // 8, block=512, bits=8),
    qgz=QgZ(nodes=1, gpus_per_node=8, bucket=LLAMA_PHI, block=512, bits=4),
)

TWO_HOP = Workload(
    "two-hop bucket: 2^28 per rank, N_d=16 (2x8), int4 B=256, Student-t(3) grads with outliers",
    qwz=None,
    qgz=QgZ(nodes=2, gpus_per_node=8, bucket=1 << 28, block=256, bits=4,
            grad=GRAD_T3_OUTLIERS),
)

SEVEN_B_PHI = 7 * 10 ** 9
SEVEN_B = Workload(
    "7B: qwZ int8 B=2048 over 7e9 weights in 2^28 chunks; qgZ N_d=64 (8x8) bucket 2^26 "
    "int4 B=256; fused Adam 2^26; standalone Adam 109,375,000",
    qwz=QwZ(nranks=1, shard=1 << 28, block=2048, bits=8,
            calls=-(-SEVEN_B_PHI // (1 << 28)),
            tail_shard=SEVEN_B_PHI - (SEVEN_B_PHI // (1 << 28)) * (1 << 28)),
    qgz=QgZ(nodes=8, gpus_per_node=8, bucket=1 << 26, block=256, bits=4),
    standalone_adam=SEVEN_B_PHI // 64,
)

WORKLOADS = {"tiny": TINY, "llama": LLAMA, "two_hop": TWO_HOP, "7b": SEVEN_B}

SWEEP_BLOCKS = (64, 256, 1024, 4096)
SWEEP_BITS = (8, 4)
SWEEP_TOPOS = ((1, 8), (4, 8), (16, 8))
SWEEP_MIB = (1, 4, 16, 64, 256, 1024)


def sweep_points():
    """The 144 sweep points in nested order (block, bits, topology, message);
    the seed of a point is its index.  The message size counts the bf16 input
    bytes of one rank's bucket, so bucket = MiB * 2**19 elements."""
    i = 0
    for block in SWEEP_BLOCKS:
        for bits in SWEEP_BITS:
            for nodes, g in SWEEP_TOPOS:
                for mib in SWEEP_MIB:
                    bucket = mib << 19
                    yield i, Workload(
                        f"sweep#{i}: B={block} int{bits} N_d={nodes * g} ({nodes}x{g}) "
                        f"{mib} MiB/rank",
                        qwz=QwZ(nranks=nodes * g, shard=bucket, block=block, bits=bits),
                        qgz=QgZ(nodes=nodes, gpus_per_node=g, bucket=bucket, block=block,
                                bits=bits),
                        fused_adam=False, seed=i)
                    i += 1


def scaled(wl: Workload, factor: int) -> Workload:
    """The same workload with every shard and bucket divided by `factor`
    (rounded down to whole blocks per slice): a smaller instance for profiling."""
    import dataclasses
    q, g = wl.qwz, wl.qgz
    if q is not None:
        shard = max(q.block, (q.shard // factor) // q.block * q.block)
        q = dataclasses.replace(q, shard=shard, calls=1, tail_shard=0)
    if g is not None:
        unit = g.nd * g.block
        g = dataclasses.replace(g, bucket=max(unit, (g.bucket // factor) // unit * unit))
    return dataclasses.replace(wl, name=f"{wl.name} / {factor}", qwz=q, qgz=g)
