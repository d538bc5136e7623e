"""Device buffers and call sequence of one pass of the ZeRO++ data-parallel path.

Plumbing only: allocates the simulated ranks' buffers with torch and issues
the C-ABI calls in order.  One pass (``CodecPath.run``) is

  qwZ   zpp_qwz_quant (every rank's weight shard) -> zpp_qwz_dequant (the
        all-gather receiver, one full bf16 copy), optionally over several
        chunks of a long weight tensor;
  hpZ   optionally the backward all-gather from the node's secondary
        partitions (zpp_hpz_gather): local rank l keeps the received messages
        of shards l*N .. l*N + N - 1, and the backward pass re-gathers the
        weights from those G buffers into the same workspace;
  qgZ   zpp_qgz_reorder_quant (every rank's bucket) -> zpp_qgz_hop_reduce(1)
        -> zpp_qgz_hop_reduce(2) when there is more than one node, the final
        hop applying the Adam step to every rank's owned slice.  With M > 1
        micro-batches the first M-1 are summed by zpp_grad_accumulate into an
        fp32 accumulator and the one-shot quantizer reads accumulator + last
        micro-batch (zpp_qgz_reorder_quant_acc).
  Adam  optionally zpp_shard_adam_step over a further owned shard (the part
        of a rank's parameters outside the reduced bucket).
  ring  the comparator: the qgZ chain replaced by a ring reduce-scatter of
        quantized gradients (N_d zpp_ring_rs_step launches, a requantization
        at every hop) and zpp_shard_adam_step on the reduced gradient.

Every message between two calls is a separate HBM buffer, as the wire
between two GPUs would be.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib as Z


@dataclass(frozen=True)
class QwzSpec:
    nranks: int
    shard: int
    block: int
    bits: int = 8
    chunks: int = 1          # the weight tensor is `chunks` calls of nranks*shard
    tail_shard: int = 0      # shard of the last call when nonzero
    nodes: int = 1           # hpZ: the nranks ranks are `nodes` nodes of nranks/nodes GPUs

    def call_shards(self):
        s = [self.shard] * self.chunks
        if self.tail_shard:
            s[-1] = self.tail_shard
        return s

    @property
    def phi(self):
        return self.nranks * sum(self.call_shards())


@dataclass(frozen=True)
class QgzSpec:
    nodes: int
    gpus_per_node: int
    bucket: int
    block: int
    bits: int = 4

    @property
    def nd(self):
        return self.nodes * self.gpus_per_node

    @property
    def L(self):
        return self.bucket // self.nd


@dataclass(frozen=True)
class AdamSpec:
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    step: int = 1

    def hparams(self):
        return (self.lr, self.beta1, self.beta2, self.eps, self.step)


def _empty(n, dtype, device):
    return torch.empty(int(n), dtype=dtype, device=device)


class CodecPath:
    """Buffers of one simulated ZeRO++ step on one device.

    Inputs the caller fills: ``w`` (bf16 weights, all calls concatenated),
    ``grads`` (bf16 [N_d][bucket]; with micro-batches every tensor of
    ``grads_mb``) and the Adam state ``master, m, v``
    (fp32 [bucket], element r*L + i owned by rank r).
    """

    def __init__(self, qwz: QwzSpec | None, qgz: QgzSpec | None, adam: AdamSpec | None,
                 device="cuda", keep_grad: bool = False, write_param: bool = True,
                 fuse_qwz: bool = False, microbatches: int = 1, standalone_adam: int = 0,
                 hpz: bool = False, ring: bool = False):
        """ring: reduce the gradients with the quantized ring instead of qgZ
        (no micro-batches, no fused qwZ).
        hpz: after the forward gather, the backward gather of the weights
        from the secondary partitions (qwZ with one call, nranks divisible by
        the node count).
        standalone_adam: parameters of a separate owned shard stepped by
        zpp_shard_adam_step after the reduce (fp32 ``sa_grad``, ``sa_master``,
        ``sa_m``, ``sa_v``, bf16 ``sa_param``).
        microbatches: gradients of that many micro-batches (``grads_mb``,
        ``grads`` being the last) are accumulated before the reduce.
        fuse_qwz: the weights' qwZ message is produced by the final hop's
        Adam pass from the new parameters (zpp_qgz_final_hop_adam_qwz) instead
        of a separate quantize call; needs the qwZ shards to be the ranks'
        owned qgZ slices (nranks = N_d, shard = L, same block, int8)."""
        self.qwz, self.qgz, self.adam = qwz, qgz, adam
        self.fuse_qwz = fuse_qwz
        if microbatches < 1:
            raise ValueError("microbatches must be >= 1")
        self.microbatches = microbatches
        if fuse_qwz:
            ok = (qwz is not None and qgz is not None and adam is not None and qwz.bits == 8
                  and qwz.chunks == 1 and qwz.nranks == qgz.nd and qwz.shard == qgz.L
                  and qwz.block == qgz.block)
            if not ok:
                raise ValueError("fuse_qwz needs qwZ shards equal to the owned qgZ slices")
        self.hpz = hpz
        self.ring = ring
        if ring and (qgz is None or microbatches > 1 or fuse_qwz):
            raise ValueError("ring replaces a plain qgZ chain")
        if hpz and (qwz is None or qwz.chunks != 1 or qwz.nranks % qwz.nodes):
            raise ValueError("hpz needs one qwZ call over nodes x GPUs-per-node shards")
        self.device = torch.device(device)
        dev = self.device
        self.launches_per_run = 0
        if qwz is not None:
            self.w = _empty(qwz.phi, torch.bfloat16, dev)
            shards = qwz.call_shards()
            self.w_codes = [_empty(qwz.nranks * Z.zpp_codes_bytes(s, qwz.bits), torch.uint8, dev)
                            for s in sorted(set(shards))]
            self._codes_of = {s: i for i, s in enumerate(sorted(set(shards)))}
            self.w_scales = [_empty(qwz.nranks * Z.zpp_num_blocks(s, qwz.block), torch.float32, dev)
                             for s in sorted(set(shards))]
            self.w_full = _empty(qwz.phi, torch.bfloat16, dev)
            self.launches_per_run += (1 if fuse_qwz else 2) * len(shards) + (1 if hpz else 0)
        if qgz is not None:
            nd, b = qgz.nd, qgz.bucket
            self.grads_mb = [_empty(nd * b, torch.bfloat16, dev) for _ in range(microbatches)]
            self.grads = self.grads_mb[-1]
            self.acc = _empty(nd * b, torch.float32, dev) if microbatches > 1 else None
            self.launches_per_run += microbatches - 1
            if ring:
                L = qgz.L
                self.ring_msgs = [(_empty(nd * Z.zpp_codes_bytes(L, qgz.bits), torch.uint8, dev),
                                   _empty(nd * (L // qgz.block), torch.float32, dev))
                                  for _ in range(2)]
                self.launches_per_run += nd + (1 if adam is not None else 0)
            else:
                self.msg1 = _empty(nd * Z.zpp_codes_bytes(b, qgz.bits), torch.uint8, dev)
                self.msg1_scales = _empty(nd * (b // qgz.block), torch.float32, dev)
                self.launches_per_run += 2
            if qgz.nodes > 1 and not ring:
                nl = qgz.nodes * qgz.L
                self.msg2 = _empty(nd * Z.zpp_codes_bytes(nl, qgz.bits), torch.uint8, dev)
                self.msg2_scales = _empty(nd * (nl // qgz.block), torch.float32, dev)
                self.launches_per_run += 1
            self.grad_out = _empty(b, torch.float32, dev) \
                if (keep_grad or adam is None or ring) else None
            if adam is not None:
                self.master = _empty(b, torch.float32, dev)
                self.m = torch.zeros(b, dtype=torch.float32, device=dev)
                self.v = torch.zeros(b, dtype=torch.float32, device=dev)
                self.param = _empty(b, torch.bfloat16, dev) if write_param else None
        self.standalone_adam = int(standalone_adam)
        if self.standalone_adam:
            if adam is None:
                raise ValueError("standalone_adam needs the Adam hyper-parameters")
            n = self.standalone_adam
            self.sa_grad = _empty(n, torch.float32, dev)
            self.sa_master = _empty(n, torch.float32, dev)
            self.sa_m = torch.zeros(n, dtype=torch.float32, device=dev)
            self.sa_v = torch.zeros(n, dtype=torch.float32, device=dev)
            self.sa_param = _empty(n, torch.bfloat16, dev) if write_param else None
            self.launches_per_run += 1

    # ---- the pass ---------------------------------------------------------------
    # `mark(name)`, when given, is called after each launch (the bench records a
    # CUDA event there to time every kernel of the pass).
    def prime_fused_qwz(self, stream=None):
        """Fused mode: the first step's weight message, from the initial weights."""
        q = self.qwz
        Z.zpp_qwz_quant(self.w, q.nranks, q.shard, q.block, q.bits, self.w_codes[0],
                        self.w_scales[0], stream)

    def run_qwz(self, stream=None, mark=None):
        q = self.qwz
        if self.fuse_qwz:  # the message was written by the previous step's Adam pass
            Z.zpp_qwz_dequant(self.w_codes[0], self.w_scales[0], q.nranks, q.shard, q.block,
                              q.bits, self.w_full, stream)
            if mark:
                mark("qwz_dequant")
            return
        off = 0
        for s in q.call_shards():
            n = q.nranks * s
            i = self._codes_of[s]
            x = self.w[off:off + n]
            Z.zpp_qwz_quant(x, q.nranks, s, q.block, q.bits, self.w_codes[i], self.w_scales[i],
                            stream)
            if mark:
                mark("qwz_quant")
            Z.zpp_qwz_dequant(self.w_codes[i], self.w_scales[i], q.nranks, s, q.block, q.bits,
                              self.w_full[off:off + n], stream)
            if mark:
                mark("qwz_dequant")
            off += n

    def secondary_partitions(self):
        """(codes, scales) views of every local rank's secondary partition:
        the received messages of its N shards, kept from the forward gather."""
        q = self.qwz
        N, G = q.nodes, q.nranks // q.nodes
        cb, nb = Z.zpp_codes_bytes(q.shard, q.bits), Z.zpp_num_blocks(q.shard, q.block)
        c, s = self.w_codes[0], self.w_scales[0]
        return ([c[l * N * cb:(l + 1) * N * cb] for l in range(G)],
                [s[l * N * nb:(l + 1) * N * nb] for l in range(G)])

    def run_hpz(self, stream=None, mark=None):
        q = self.qwz
        codes, scales = self.secondary_partitions()
        Z.zpp_hpz_gather(q.nranks // q.nodes, q.nodes, q.shard, q.block, q.bits, codes, scales,
                         self.w_full, stream)
        if mark:
            mark("hpz_gather")

    def run_ring(self, stream=None, adam_step: int | None = None, mark=None):
        g = self.qgz
        nd = g.nd
        for step in range(nd):
            ci, si = self.ring_msgs[(step + 1) & 1] if step else (None, None)
            co, so = self.ring_msgs[step & 1] if step < nd - 1 else (None, None)
            Z.zpp_ring_rs_step(step, nd, g.bucket, g.block, g.bits, self.grads, ci, si, co, so,
                               self.grad_out if step == nd - 1 else None, stream)
            if mark:
                mark("ring_step")
        if self.adam is not None:
            hp = list(self.adam.hparams())
            if adam_step is not None:
                hp[4] = adam_step
            Z.zpp_shard_adam_step(self.grad_out, g.bucket, tuple(hp),
                                  (self.master, self.m, self.v, self.param), stream)
            if mark:
                mark("ring_adam")

    def run_qgz(self, stream=None, adam_step: int | None = None, mark=None):
        g = self.qgz
        if self.ring:
            return self.run_ring(stream, adam_step, mark)
        if self.microbatches > 1:
            n = g.nd * g.bucket
            for k, gk in enumerate(self.grads_mb[:-1]):
                Z.zpp_grad_accumulate(gk, self.acc, n, k == 0, stream)
                if mark:
                    mark("grad_accumulate")
            Z.zpp_qgz_reorder_quant_acc(self.grads, self.acc, g.nodes, g.gpus_per_node, g.bucket,
                                        g.block, g.bits, self.msg1, self.msg1_scales, stream)
            if mark:
                mark("qgz_reorder_quant_acc")
        else:
            Z.zpp_qgz_reorder_quant(self.grads, g.nodes, g.gpus_per_node, g.bucket, g.block,
                                    g.bits, self.msg1, self.msg1_scales, stream)
            if mark:
                mark("qgz_reorder_quant")
        adam = state = None
        if self.adam is not None:
            hp = list(self.adam.hparams())
            if adam_step is not None:
                hp[4] = adam_step
            adam = tuple(hp)
            state = (self.master, self.m, self.v, self.param)
        if self.fuse_qwz:
            if g.nodes > 1:
                Z.zpp_qgz_hop_reduce(1, self.msg1, self.msg1_scales, g.nodes, g.gpus_per_node,
                                     g.bucket, g.block, g.bits, codes_out=self.msg2,
                                     scales_out=self.msg2_scales, stream=stream)
                if mark:
                    mark("qgz_hop1")
            hop, ci, si = (1, self.msg1, self.msg1_scales) if g.nodes == 1 else \
                (2, self.msg2, self.msg2_scales)
            Z.zpp_qgz_final_hop_adam_qwz(hop, ci, si, g.nodes, g.gpus_per_node, g.bucket, g.block,
                                         g.bits, self.grad_out, adam, state, 8, self.w_codes[0],
                                         self.w_scales[0], stream)
            if mark:
                mark("qgz_final_hop_qwz")
        elif g.nodes == 1:
            Z.zpp_qgz_hop_reduce(1, self.msg1, self.msg1_scales, g.nodes, g.gpus_per_node,
                                 g.bucket, g.block, g.bits, grad_out=self.grad_out, adam=adam,
                                 state=state, stream=stream)
            if mark:
                mark("qgz_final_hop")
        else:
            Z.zpp_qgz_hop_reduce(1, self.msg1, self.msg1_scales, g.nodes, g.gpus_per_node,
                                 g.bucket, g.block, g.bits, codes_out=self.msg2,
                                 scales_out=self.msg2_scales, stream=stream)
            if mark:
                mark("qgz_hop1")
            Z.zpp_qgz_hop_reduce(2, self.msg2, self.msg2_scales, g.nodes, g.gpus_per_node,
                                 g.bucket, g.block, g.bits, grad_out=self.grad_out, adam=adam,
                                 state=state, stream=stream)
            if mark:
                mark("qgz_final_hop")

    def run_standalone_adam(self, stream=None, adam_step: int | None = None, mark=None):
        hp = list(self.adam.hparams())
        if adam_step is not None:
            hp[4] = adam_step
        Z.zpp_shard_adam_step(self.sa_grad, self.standalone_adam, tuple(hp),
                              (self.sa_master, self.sa_m, self.sa_v, self.sa_param), stream)
        if mark:
            mark("shard_adam")

    def run(self, stream=None, adam_step: int | None = None, mark=None):
        if self.qwz is not None:
            self.run_qwz(stream, mark)
        if self.hpz:
            self.run_hpz(stream, mark)
        if self.qgz is not None:
            self.run_qgz(stream, adam_step, mark)
        if self.standalone_adam:
            self.run_standalone_adam(stream, adam_step, mark)

    def _bind_input_set(self, k: int, n_sets: int, names=("w", "grads_mb", "sa_grad")):
        """Point the inputs in `names` (of w / grads_mb / sa_grad; grads
        follows grads_mb) at device input set k of n_sets.  Set 0 is the
        path's own buffers; the others are allocated on first use."""
        if getattr(self, "_sets", None) is None or len(self._sets) != n_sets:
            own = {"w": getattr(self, "w", None), "grads_mb": getattr(self, "grads_mb", None),
                   "sa_grad": getattr(self, "sa_grad", None)}
            if getattr(self, "_sets", None):
                own = self._sets[0]
            self._sets = [own]
            for _ in range(1, n_sets):
                self._sets.append({
                    "w": torch.empty_like(own["w"]) if own["w"] is not None else None,
                    "grads_mb": [torch.empty_like(t) for t in own["grads_mb"]]
                    if own["grads_mb"] is not None else None,
                    "sa_grad": torch.empty_like(own["sa_grad"]) if own["sa_grad"] is not None
                    else None})
            self._last_read = {}  # (set, input) -> event after the kernels that last read it
            self._bound = {"w": 0, "grads_mb": 0, "sa_grad": 0}
            self._next_set = 0
        b = self._sets[k]
        if "w" in names and b["w"] is not None:
            self.w = b["w"]
            self._bound["w"] = k
        if "grads_mb" in names and b["grads_mb"] is not None:
            self.grads_mb = b["grads_mb"]
            self.grads = self.grads_mb[-1]
            self._bound["grads_mb"] = k
        if "sa_grad" in names and b["sa_grad"] is not None:
            self.sa_grad = b["sa_grad"]
            self._bound["sa_grad"] = k

    def run_from_host(self, w_host=None, grads_host=None, param_host=None, stream=None,
                      adam_step: int | None = None, sa_grad_host=None, sa_param_host=None,
                      copy_streams: int = 2, input_sets: int = 2):
        """One pass on host-resident data: copy this step's weights and
        gradients in from pinned host tensors, run, and copy the updated
        16-bit parameters back.  `grads_host` is one tensor, or one per
        micro-batch; `sa_grad_host`/`sa_param_host` are the standalone shard's
        fp32 gradients in and bf16 parameters out.

        The copies are split into chunks over `copy_streams` streams each way
        and overlap the kernels: the qwZ kernels start once the weights are in
        while the gradients are still arriving.  Successive calls take turns
        over `input_sets` sets of device input buffers (weights, gradients,
        standalone gradients), so with two or more sets the next call's
        inputs start arriving as soon as this call's have, under this call's
        kernels and read-back; a set is refilled only once the kernels of the
        call that last used it have read it.  After the call, `w`, `grads_mb`,
        `grads` and `sa_grad` are that call's device inputs (those not copied
        in stay where they were).  Returns the bytes moved each way
        (h2d, d2h)."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        n_cs = max(1, int(copy_streams))
        n_sets = max(1, int(input_sets))
        if getattr(self, "_copy_in", None) is None or len(self._copy_in) != n_cs:
            self._copy_in = [torch.cuda.Stream(self.device) for _ in range(n_cs)]
            self._copy_out = [torch.cuda.Stream(self.device) for _ in range(n_cs)]
        cin, cout = self._copy_in, self._copy_out
        if getattr(self, "_sets", None) is None or len(self._sets) != n_sets:
            self._bind_input_set(0, n_sets, ())
        k = self._next_set
        self._next_set = (k + 1) % n_sets
        # only the inputs this call copies in move to set k; the kernels read the rest
        # where the caller left them
        copied = [n for n, h in (("w", w_host), ("grads_mb", grads_host), ("sa_grad", sa_grad_host))
                  if h is not None]
        self._bind_input_set(k, n_sets, copied)
        h2d = d2h = 0

        def after(stream_from, streams_to):
            ev = torch.cuda.Event()
            ev.record(stream_from)
            for t in streams_to:
                t.wait_event(ev)
            return ev

        def split_copy(pairs, streams):
            """Copy every (dst, src) pair in chunks round-robin over `streams`;
            returns the bytes copied."""
            nbytes, i = 0, 0
            for dst, src in pairs:
                n = src.numel()
                nbytes += n * src.element_size()
                step = max(1 << 20, -(-n // len(streams)))
                for lo in range(0, n, step):
                    with torch.cuda.stream(streams[i % len(streams)]):
                        dst[lo:lo + step].copy_(src[lo:lo + step], non_blocking=True)
                    i += 1
            return nbytes

        # a buffer of set k is refilled once the kernels that last read it are done
        for n in copied:
            ev = self._last_read.get((k, n))
            if ev is None:
                after(s, cin)
            else:
                for c in cin:
                    c.wait_event(ev)
        if w_host is not None:
            h2d += split_copy([(self.w, w_host)], cin)
            for c in cin:
                after(c, [s])
        if self.qwz is not None:
            self.run_qwz(s.cuda_stream)
        if self.hpz:
            self.run_hpz(s.cuda_stream)
        pairs = []
        if grads_host is not None:
            hosts = grads_host if isinstance(grads_host, (list, tuple)) else [grads_host]
            if len(hosts) != self.microbatches:
                raise ValueError("grads_host: one tensor per micro-batch")
            pairs += list(zip(self.grads_mb, hosts))
        if sa_grad_host is not None:
            pairs.append((self.sa_grad, sa_grad_host))
        if pairs:
            h2d += split_copy(pairs, cin)
            for c in cin:
                after(c, [s])
        if self.qgz is not None:
            self.run_qgz(s.cuda_stream, adam_step)
        if self.standalone_adam:
            self.run_standalone_adam(s.cuda_stream, adam_step)
        read = torch.cuda.Event()
        read.record(s)
        for n, j in self._bound.items():
            self._last_read[(j, n)] = read
        back = []
        if param_host is not None:
            back.append((param_host, self.param if self.param is not None else self.master))
        if sa_param_host is not None:
            back.append((sa_param_host, self.sa_param if self.sa_param is not None
                         else self.sa_master))
        if back:
            after(s, cout)
            d2h += split_copy(back, cout)
            for c in cout:  # the next step's Adam must not overwrite them before
                after(c, [s])
        return h2d, d2h
