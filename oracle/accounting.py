"""Byte and memory accounting of the ZeRO / ZeRO++ step (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Units: ``M`` is one 16-bit copy of the model, ``2*Phi`` bytes ("Quantized LLM
Training at Scale with ZeRO++", section "Understanding the ZeRO-3
Communication Volume"; the ZeRO-1/2/3 page counts the same quantity as Phi).

Everything here is exact integer arithmetic on buffer sizes: element counts
times element sizes of the buffers a rank holds or sends.  Message sizes come
from the same size rules the oracle's quantizers use for their output arrays
(``codes_bytes``, ``num_blocks``), and a test checks them against the arrays
the oracle actually returns.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction

import numpy as np

from . import block_dequant, block_quant, codes_bytes, num_blocks

BF16 = 2
FP32 = 4


def quantized_bytes(n: int, block: int, bits: int) -> int:
    """Bytes of one block-quantized message of n elements: codes + fp32 scales."""
    return codes_bytes(n, bits) + FP32 * num_blocks(n, block)


# ---- communication volume per iteration, in units of M -----------------------

def zero3_volume() -> dict:
    """ZeRO-3: forward all-gather M + backward all-gather M + reduce-scatter M
    ("Quantized LLM Training at Scale with ZeRO++", ZeRO-3 volume list;
    ZeRO-1/2/3 page, Stage 3 communication: 3 Phi per GPU)."""
    return {"fwd": Fraction(1), "bwd": Fraction(1), "grad": Fraction(1), "total": Fraction(3)}


def zeropp_volume(phi: int, w_block: int, w_bits: int, g_block: int, g_bits: int) -> dict:
    """ZeRO++ per-iteration volume as fractions of M = 2*phi bytes.

    fwd  : qwZ message (codes + scales) of the whole model / 2 phi  (QWZ).
    bwd  : cross-node bytes of the backward all-gather under hpZ = 0 (HPZ: the
           secondary replica inside each node serves the backward gather).
    grad : the one-shot qgZ message of a bucket / its bf16 size (QGZ).
    """
    fwd = Fraction(quantized_bytes(phi, w_block, w_bits), BF16 * phi)
    grad = Fraction(quantized_bytes(phi, g_block, g_bits), BF16 * phi)
    bwd = Fraction(0)
    return {"fwd": fwd, "bwd": bwd, "grad": grad, "total": fwd + bwd + grad}


def cross_node_bytes(N: int, G: int, bucket: int, block: int, bits: int) -> dict:
    """Bytes one node sends to other nodes for one gradient bucket.

    two_hop: after hop 1 each rank holds N slots of L elements and sends the
             N-1 foreign slots across nodes.
    flat   : a single all-to-all of the one-shot message sends every slice
             owned by a rank of another node, from every rank of the node.
    """
    Nd = N * G
    L = bucket // Nd
    slot = quantized_bytes(L, block, bits)
    two_hop = G * (N - 1) * slot
    flat = G * (Nd - G) * slot
    return {"two_hop": two_hop, "flat": flat}


# ---- per-rank memory ---------------------------------------------------------

@dataclass(frozen=True)
class Buffer:
    name: str
    elems: Fraction
    elem_bytes: int

    @property
    def nbytes(self) -> Fraction:
        return self.elems * self.elem_bytes


def rank_buffers(stage: int, phi: int, nd: int) -> list[Buffer]:
    """Persistent per-rank buffers of mixed-precision Adam training.

    16-bit params (2 B), 16-bit grads (2 B), fp32 master, m, v (4 B each),
    "ZeRO-1/2/3" page, the 16 B/param breakdown; stage 0 is plain data
    parallelism.  Transient buckets are not counted (the Stage-2 page notes
    that bucketing frees gradient memory progressively).
    """
    full, shard = Fraction(phi), Fraction(phi, nd)
    p = full if stage < 3 else shard
    g = full if stage < 2 else shard
    o = full if stage < 1 else shard
    return [Buffer("param16", p, BF16), Buffer("grad16", g, BF16),
            Buffer("master32", o, FP32), Buffer("m32", o, FP32), Buffer("v32", o, FP32)]


def rank_memory(stage: int, phi: int, nd: int) -> Fraction:
    return sum((b.nbytes for b in rank_buffers(stage, phi, nd)), Fraction(0))


# ---- O8: block vs global quantization error ------------------------------------

def quant_errors(x: np.ndarray, block: int, bits: int) -> dict:
    """RMSE and max-abs error of block and of global (one-scale) quantization.

    Pinned by the invariant block RMSE <= global RMSE.  The talk's 3.3x
    precision figure is parity unpinned: the pages give neither its data nor
    its metric, so the ratio is only reported."""
    x = np.asarray(x, dtype=np.float32).reshape(-1)
    out = {}
    for name, b in (("block", block), ("global", max(x.size, 1))):
        c, s = block_quant(x, b, bits)
        y = block_dequant(c, s, x.size, b, bits)
        e = y.astype(np.float64) - x.astype(np.float64)
        out[name] = {"rmse": float(np.sqrt(np.mean(e * e))), "max": float(np.max(np.abs(e)))}
    out["rmse_ratio"] = out["global"]["rmse"] / max(out["block"]["rmse"], 1e-300)
    out["max_ratio"] = out["global"]["max"] / max(out["block"]["max"], 1e-300)
    return out
