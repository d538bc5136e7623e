"""Complete comparison of full-size GPU outputs with the oracle.

Every output element of a full-size pass is compared, not a sample: the
outputs are copied to the host once, and the oracle recomputes them in
independent pieces that run side by side on the host cores (each piece is the
single-threaded C oracle on its own inputs, regenerated on the host by the
counter-based generator):

* qwZ: blocks restart at every shard and are independent, so a shard splits
  at any block boundary into pieces the oracle quantizes on their own.
* qgZ: blocks never straddle slices, so the block positions [b0, b1) of every
  slice of every rank form a self-contained smaller bucket ("mini bucket") of
  N_d slices of (b1 - b0) * B elements: its one-shot messages, hop-1 messages,
  reduced gradient and Adam state are exactly those block positions of the
  full pass.  The groups of block positions cover every block.
* The ring comparator: blocks restart at chunk starts, so the same grouping
  applies to it.
* Adam is elementwise.

Test infrastructure only (imported by the GPU tests).
"""
from __future__ import annotations

import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import synth
from synth import workloads as W
from gpu_helpers import GRAD_RTOL

WORKERS = max(1, min(64, os.cpu_count() or 1))
GROUP_ELEMS = 1 << 25      # input elements of one qgZ piece (all ranks)
QWZ_PIECE = 1 << 24        # weight elements of one qwZ piece
_pool = None


def pool() -> ThreadPoolExecutor:
    global _pool
    if _pool is None:
        _pool = ThreadPoolExecutor(max_workers=WORKERS)
    return _pool


_tls = threading.local()


def scratch(name, shape, dtype) -> np.ndarray:
    """A per-thread host buffer reused across pieces (fresh pages are costly)."""
    bufs = getattr(_tls, "bufs", None)
    if bufs is None:
        bufs = _tls.bufs = {}
    n = int(np.prod(shape))
    b = bufs.get((name, np.dtype(dtype).str))
    if b is None or b.size < n:
        b = np.empty(n, dtype)
        bufs[(name, np.dtype(dtype).str)] = b
    return b[:n].reshape(shape)


def host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> host numpy array (uint16 for 16-bit tensors)."""
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.view(torch.int16)
        return t.cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _first_bad(got, want):
    got, want = np.asarray(got), np.asarray(want)
    if got.shape != want.shape:
        return f"shape {got.shape} != {want.shape}"
    bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
    if bad.size == 0:
        return None
    g, w = got.reshape(-1), want.reshape(-1)
    return f"{bad.size} mismatches, first at flat {bad[:3]}: got {g[bad[:3]]} want {w[bad[:3]]}"


def eq_bytes(got, want, what, fails):
    msg = _first_bad(got, want)
    if msg:
        fails.append(f"{what}: {msg}")


def eq_f32(got, want, what, fails):
    eq_bytes(np.ascontiguousarray(got, np.float32).view(np.uint32),
             np.ascontiguousarray(want, np.float32).view(np.uint32), what, fails)


def _same_f32(got, want):
    got, want = np.asarray(got), np.asarray(want)
    return got.shape == want.shape and np.array_equal(
        np.ascontiguousarray(got, np.float32).view(np.uint32),
        np.ascontiguousarray(want, np.float32).view(np.uint32))


def close_rel(got, want, rtol, what, fails):
    if _same_f32(got, want):    # bit-identical (the usual case) is within any tolerance
        return
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    ok = np.abs(got - want) <= rtol * np.abs(want) + 1e-30
    if not ok.all():
        fails.append(f"{what}: {np.count_nonzero(~ok)} outside {rtol} relative")


def close_grad(got, want, block, what, fails):
    if _same_f32(got, want):
        return
    got = np.asarray(got, np.float64).reshape(-1, block)
    want = np.asarray(want, np.float64).reshape(-1, block)
    tol = GRAD_RTOL * np.abs(want).max(axis=1, keepdims=True)
    if not np.all(np.abs(got - want) <= tol):
        fails.append(f"{what}: outside {GRAD_RTOL} of the block maximum")


def bf16_ulp(got_u16, want_u16, what, fails, ulp=1):
    if np.array_equal(np.asarray(got_u16), np.asarray(want_u16)):
        return

    def key(u):
        u = np.asarray(u, np.uint16).astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), u + 0x8000)
    d = np.abs(key(got_u16) - key(want_u16))
    if d.max(initial=0) > ulp:
        fails.append(f"{what}: max {d.max()} ulp")


def widen(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def gather(jobs) -> list[str]:
    """Run fn() for every job on the pool; every job returns its list of
    failures."""
    fails = []
    for f in [pool().submit(j) for j in jobs]:
        fails += f.result()
    return fails


def assert_no_failures(fails, what):
    assert not fails, f"{what}: {len(fails)} failing pieces; first: " + " | ".join(fails[:4])


# ---- qwZ ------------------------------------------------------------------------------

def qwz_jobs(codes, scales, y, nranks, shard, block, bits, seed, gstart, tag):
    """Pieces checking one call: codes [nranks][codes_bytes(shard)], scales
    [nranks][num_blocks(shard)], y [nranks][shard] (host arrays, any of them
    None to skip), the weights starting at global index gstart."""
    cb, nb = oracle.codes_bytes(shard, bits), oracle.num_blocks(shard, block)
    piece = max(block, QWZ_PIECE // block * block)
    jobs = []
    for r in range(nranks):
        for e0 in range(0, shard, piece):
            e1 = min(shard, e0 + piece)

            def job(r=r, e0=e0, e1=e1):
                fails = []
                n = e1 - e0
                x = synth.fill_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, gstart + r * shard + e0, n)
                wc, ws = oracle.qwz_quant(x, 1, n, block, bits)
                where = f"{tag} rank {r} elements [{e0}, {e1})"
                if codes is not None:
                    c0 = r * cb + (e0 * bits) // 8
                    eq_bytes(codes[c0:c0 + wc.size], wc, f"qwZ codes {where}", fails)
                if scales is not None:
                    s0 = r * nb + e0 // block
                    eq_f32(scales[s0:s0 + ws.size], ws, f"qwZ scales {where}", fails)
                if y is not None:
                    wy = oracle.qwz_dequant(wc, ws, 1, n, block, bits)
                    eq_bytes(y[r * shard + e0:r * shard + e1], wy, f"qwZ dequant {where}", fails)
                return fails
            jobs.append(job)
    return jobs


class QwzCapture:
    """`mark` hook of CodecPath.run / run_qwz: after every call's dequantize,
    copies that call's codes, scales and dequantized weights to the host and
    queues their complete check (the calls of a long weight tensor reuse one
    code buffer, so each is checked before the next call overwrites it)."""

    def __init__(self, path, wl, check_codes=True, max_pending=4):
        self.path, self.wl = path, wl
        self.check_codes = check_codes
        self.shards = path.qwz.call_shards()
        self.call, self.off = 0, 0
        self.pending, self.max_pending = [], max_pending
        self.fails = []

    def __call__(self, name):
        if name != "qwz_dequant":
            return
        p, q = self.path, self.path.qwz
        s = self.shards[self.call]
        n = q.nranks * s
        i = p._codes_of[s]
        if torch.cuda.is_available():
            torch.cuda.synchronize()
        y = host(p.w_full[self.off:self.off + n])
        c = host(p.w_codes[i]) if self.check_codes else None
        sc = host(p.w_scales[i]) if self.check_codes else None
        jobs = qwz_jobs(c, sc, y, q.nranks, s, q.block, q.bits, self.wl.seed, self.off,
                        f"call {self.call}")
        self.pending.append([pool().submit(j) for j in jobs])
        while len(self.pending) > self.max_pending:
            self._drain_one()
        self.call += 1
        self.off += n

    def _drain_one(self):
        for f in self.pending.pop(0):
            self.fails += f.result()

    def finish(self):
        while self.pending:
            self._drain_one()
        assert self.call == len(self.shards), (self.call, len(self.shards))
        assert_no_failures(self.fails, "qwZ")


# ---- qgZ -------------------------------------------------------------------------------

def block_groups(nblk, per_group_blocks):
    per = max(1, per_group_blocks)
    return [(b0, min(nblk, b0 + per)) for b0 in range(0, nblk, per)]


def qgz_host_outputs(path):
    """The qgZ chain's outputs on the host, shaped by rank / slice position."""
    g = path.qgz
    Nd, L, B, bits, N = g.nd, g.L, g.block, g.bits, g.nodes
    cbs = (L * bits) // 8
    out = {"msg1": host(path.msg1).reshape(Nd, Nd, cbs),
           "sc1": host(path.msg1_scales).reshape(Nd, Nd, L // B)}
    if N > 1:
        out["msg2"] = host(path.msg2).reshape(Nd, N, cbs)
        out["sc2"] = host(path.msg2_scales).reshape(Nd, N, L // B)
    if path.grad_out is not None:
        out["grad"] = host(path.grad_out).reshape(Nd, L)
    if path.adam is not None:
        out["master"] = host(path.master).reshape(Nd, L)
        out["m"] = host(path.m).reshape(Nd, L)
        out["v"] = host(path.v).reshape(Nd, L)
        if path.param is not None:
            out["param"] = host(path.param).reshape(Nd, L)
    if path.microbatches > 1:
        out["acc"] = host(path.acc).reshape(Nd, Nd, L)
    if path.fuse_qwz:
        out["wc"] = host(path.w_codes[0]).reshape(Nd, L)
        out["ws"] = host(path.w_scales[0]).reshape(Nd, L // B)
    return out


def check_qgz_complete(path, wl, adam_step=None):
    """Every one-shot code and scale, hop-1 code and scale, accumulator value,
    reduced-gradient float, Adam element and fused qwZ code of a full pass
    (m = v = 0 before the step, master = the widened weights)."""
    g = path.qgz
    N, G, Nd, L, B, bits = g.nodes, g.gpus_per_node, g.nd, g.L, g.block, g.bits
    recipe = wl.qgz.grad
    M = path.microbatches
    seed = wl.seed
    out = qgz_host_outputs(path)
    bb = (B * bits) // 8
    groups = block_groups(L // B, GROUP_ELEMS // (Nd * Nd * B))
    a = wl.adam
    step = a.step if adam_step is None else adam_step

    def job(b0, b1):
        fails = []
        Lm = (b1 - b0) * B
        tag = f"block positions [{b0}, {b1})"
        mbs = []
        for k in range(M):
            mini = scratch(f"mini{k}", (Nd, Nd, Lm), np.uint16)
            for r in range(Nd):
                s = synth.grad_stream(r, k)
                for j in range(Nd):
                    synth.fill_u16(recipe, seed, s, j * L + b0 * B, Lm, out=mini[r, j])
            mbs.append(mini.reshape(-1))
        bucket_m = Nd * Lm
        if M == 1:
            c1, s1 = oracle.qgz_reorder_quant(mbs[0], N, G, bucket_m, B, bits)
        else:
            wa = oracle.grad_accumulate(mbs[:-1])
            eq_f32(out["acc"][:, :, b0 * B:b1 * B], wa.reshape(Nd, Nd, Lm), f"accumulator {tag}",
                   fails)
            c1, s1 = oracle.qgz_reorder_quant_f32(oracle.grad_accumulate(mbs), N, G, bucket_m, B,
                                                  bits)
        del mbs
        eq_bytes(out["msg1"][:, :, b0 * bb:b1 * bb], c1.reshape(Nd, Nd, -1),
                 f"one-shot codes {tag}", fails)
        eq_f32(out["sc1"][:, :, b0:b1], s1.reshape(Nd, Nd, -1), f"one-shot scales {tag}", fails)
        if N == 1:
            gref = oracle.qgz_hop1(c1, s1, N, G, bucket_m, B, bits)
        else:
            c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket_m, B, bits)
            eq_bytes(out["msg2"][:, :, b0 * bb:b1 * bb], c2.reshape(Nd, N, -1),
                     f"hop-1 codes {tag}", fails)
            eq_f32(out["sc2"][:, :, b0:b1], s2.reshape(Nd, N, -1), f"hop-1 scales {tag}", fails)
            gref = oracle.qgz_hop2(c2, s2, N, G, bucket_m, B, bits)
        gref = gref.reshape(Nd, Lm)
        if "grad" in out:
            got = out["grad"][:, b0 * B:b1 * B]
            close_grad(got, gref, B, f"reduced gradient {tag}", fails)
            eq_f32(got, gref, f"reduced gradient (bit-exact) {tag}", fails)
        if path.adam is not None:
            w = scratch("w", (Nd, Lm), np.uint16)
            for d in range(Nd):
                synth.fill_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, d * L + b0 * B, Lm, out=w[d])
            p0 = widen(w).reshape(-1)
            z = np.zeros(Nd * Lm, np.float32)
            wp, wm, wv, wb = oracle.adam_step(gref.reshape(-1), p0, z, z, a.lr, a.beta1, a.beta2,
                                              a.eps, step)
            sl = np.s_[:, b0 * B:b1 * B]
            close_rel(out["master"][sl], wp.reshape(Nd, Lm), 1e-5, f"master {tag}", fails)
            close_rel(out["m"][sl], wm.reshape(Nd, Lm), 1e-5, f"m {tag}", fails)
            close_rel(out["v"][sl], wv.reshape(Nd, Lm), 1e-5, f"v {tag}", fails)
            if "param" in out:
                bf16_ulp(out["param"][sl], wb.reshape(Nd, Lm), f"param {tag}", fails)
            if path.fuse_qwz:
                wc, ws = oracle.qwz_quant(wb, Nd, Lm, B, 8)
                eq_bytes(out["wc"][sl], wc.reshape(Nd, Lm), f"fused qwZ codes {tag}", fails)
                eq_f32(out["ws"][:, b0:b1], ws.reshape(Nd, -1), f"fused qwZ scales {tag}", fails)
        return fails

    fails = gather([lambda b0=b0, b1=b1: job(b0, b1) for b0, b1 in groups])
    assert_no_failures(fails, f"qgZ {Nd} ranks ({N}x{G}) L={L} B={B} int{bits}")
    return len(groups)


def check_ring_complete(grad_dev, qgz: W.QgZ, seed):
    """Every reduced-gradient float of the quantized ring over the whole
    bucket (blocks restart at chunk starts)."""
    nd, L, B, bits = qgz.nd, qgz.slice_elems, qgz.block, qgz.bits
    grad = host(grad_dev).reshape(nd, L)
    groups = block_groups(L // B, GROUP_ELEMS // (nd * nd * B))

    def job(b0, b1):
        fails = []
        Lm = (b1 - b0) * B
        mini = scratch("mini", (nd, nd, Lm), np.uint16)
        for r in range(nd):
            s = synth.grad_stream(r)
            for c in range(nd):
                synth.fill_u16(qgz.grad, seed, s, c * L + b0 * B, Lm, out=mini[r, c])
        want = oracle.ring_reduce_scatter(mini.reshape(-1), nd, nd * Lm, B, bits)
        eq_f32(grad[:, b0 * B:b1 * B], want.reshape(nd, Lm),
               f"ring gradient block positions [{b0}, {b1})", fails)
        return fails

    fails = gather([lambda b0=b0, b1=b1: job(b0, b1) for b0, b1 in groups])
    assert_no_failures(fails, "ring")


def check_adam_complete(dev, n, seed, hp, grad_recipe, grad_stream, master_start=0,
                        moments=True):
    """Every element of a standalone Adam step over n parameters whose
    gradient and master were drawn by synth and widened to fp32 (grad from
    (grad_recipe, grad_stream), master from the weights at master_start + i)
    and whose m and v came from their moment streams (moments) or were 0.
    `dev`: the (master, m, v, param) device tensors after the step."""
    master, m, v, param = (host(t) for t in dev)
    lr, b1, b2, eps, t = hp
    piece = 1 << 22

    def job(e0, e1):
        fails = []
        k = e1 - e0
        g = widen(synth.fill_u16(grad_recipe, seed, grad_stream, e0, k))
        p0 = widen(synth.fill_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, master_start + e0, k))
        if moments:
            m0 = widen(synth.fill_u16(W.MOMENT_M_RECIPE, seed, synth.MOMENT_M, e0, k))
            v0 = widen(synth.fill_u16(W.MOMENT_V_RECIPE, seed, synth.MOMENT_V, e0, k))
        else:
            m0 = v0 = np.zeros(k, np.float32)
        wp, wm, wv, wb = oracle.adam_step(g, p0, m0, v0, lr, b1, b2, eps, t)
        tag = f"elements [{e0}, {e1})"
        close_rel(master[e0:e1], wp, 1e-5, f"master {tag}", fails)
        close_rel(m[e0:e1], wm, 1e-5, f"m {tag}", fails)
        close_rel(v[e0:e1], wv, 1e-5, f"v {tag}", fails)
        bf16_ulp(param[e0:e1], wb, f"param {tag}", fails)
        return fails

    fails = gather([lambda e0=e0: job(e0, min(n, e0 + piece)) for e0 in range(0, n, piece)])
    assert_no_failures(fails, "standalone Adam")
