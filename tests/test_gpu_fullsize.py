"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times (CodecPath): every output element is compared with the oracle.

Inputs are generated on the device by the counter-based generator; the host
regenerates them and the oracle recomputes the outputs in independent pieces
side by side on the host cores (tests/fullcheck.py: qwZ shards split at block
boundaries; for qgZ and the ring, groups of block positions of every slice of
every rank form self-contained smaller buckets).

The sweep's 144 points are all run: completely where N_d * bucket <= 2^30
elements, and above that on sampled blocks (first, last and seeded random
blocks of every slice and shard; a sampled block position b of every slice is
a self-contained sub-problem, so the oracle runs the whole chain on the
"mini bucket" of the sampled blocks).  A point too large for one pass runs
its qgZ chain and its qwZ calls separately; a point is skipped only when its
qgZ chain alone does not fit in device memory, and the skip says so.
"""
import numpy as np
import pytest
import torch

import fullcheck as F
import oracle
import synth
from synth import workloads as W
from gpu_helpers import (assert_bf16_ulp, assert_bytes_equal, assert_f32_bitexact,
                         assert_grad_close, assert_rel_close, grads_for, zpp)

COMPLETE_MAX_ELEMS = 1 << 30   # sweep points checked completely up to this N_d * bucket

pytestmark = pytest.mark.gpu


def gather_bytes(t: torch.Tensor, starts, length):
    """Bytes [s, s + length) of a flat uint8 device tensor for every start s."""
    idx = (torch.as_tensor(np.asarray(starts, np.int64))[:, None]
           + torch.arange(length, dtype=torch.int64)[None, :]).reshape(-1).to(t.device)
    return t.index_select(0, idx).cpu().numpy()


def gather_f32(t: torch.Tensor, idx):
    return t.index_select(0, torch.as_tensor(np.asarray(idx, np.int64)).to(t.device)).cpu().numpy()


def gather_u16(t: torch.Tensor, idx):
    v = t.index_select(0, torch.as_tensor(np.asarray(idx, np.int64)).to(t.device))
    return synth.bf16_to_u16(v)


def sample_blocks(nblocks, k, seed):
    rng = np.random.default_rng(seed)
    picks = {0, nblocks - 1}
    picks.update(int(x) for x in rng.integers(0, nblocks, size=k))
    return sorted(picks)


def build_path(Z, wl: W.Workload, keep_grad=True, fuse_qwz=False, microbatches=1,
               standalone=False):
    q, g = wl.qwz, wl.qgz
    qs = gs = None
    if q is not None:
        qs = Z.QwzSpec(q.nranks, q.shard, q.block, q.bits, chunks=q.calls, tail_shard=q.tail_shard)
    if g is not None:
        gs = Z.QgzSpec(g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    a = wl.adam
    adam = Z.AdamSpec(a.lr, a.beta1, a.beta2, a.eps, a.step) if (g and wl.fused_adam) else None
    sa = wl.standalone_adam if (standalone and adam is not None) else 0
    path = Z.CodecPath(qs, gs, adam, device="cuda", keep_grad=keep_grad, fuse_qwz=fuse_qwz,
                       microbatches=microbatches, standalone_adam=sa)
    if q is not None:
        synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, qs.phi, out=path.w)
    if g is not None:
        for k, t in enumerate(path.grads_mb):
            grads_for(g, wl.seed, microbatch=k, out=t)
        if adam is not None:
            m = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, g.bucket, device="cuda")
            path.master.copy_(m.float())
            del m
    if sa:   # the bench's standalone shard: N(0, 1e-3) gradients, weights after the bucket
        t = synth.fill(W.GRAD_NORMAL, wl.seed, synth.SHARD_GRAD, 0, sa, device="cuda")
        path.sa_grad.copy_(t.float())
        synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, g.bucket, sa, out=t)
        path.sa_master.copy_(t.float())
        del t
    return path


def run_checked(path, wl, *, fused_prime=False):
    """One pass with every output compared completely with the oracle."""
    cap = F.QwzCapture(path, wl) if path.qwz is not None else None
    if fused_prime:
        path.prime_fused_qwz()
    path.run(mark=cap)
    torch.cuda.synchronize()
    if cap is not None:
        cap.finish()
    if path.qgz is not None:
        F.check_qgz_complete(path, wl)
    if path.standalone_adam:
        a = wl.adam
        F.check_adam_complete((path.sa_master, path.sa_m, path.sa_v, path.sa_param),
                              path.standalone_adam, wl.seed,
                              (a.lr, a.beta1, a.beta2, a.eps, a.step), W.GRAD_NORMAL,
                              synth.SHARD_GRAD, master_start=wl.qgz.bucket, moments=False)


def check_qwz_sampled(codes, scales, y, nranks, shard, B, bits, seed, gstart, nsample=1):
    """Sampled blocks (first, last, seeded random) of every rank's codes,
    scales and dequantized weights of one qwZ call whose weights start at
    global index gstart."""
    nb = -(-shard // B)
    cb = oracle.codes_bytes(shard, bits)
    for r in range(nranks):
        for b in sample_blocks(nb, nsample, 1000 + r):
            n = min(B, shard - b * B)
            lidx = r * shard + b * B + np.arange(n)
            x = synth.at_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, gstart + lidx)
            wc, ws = oracle.qwz_quant(x, 1, n, B, bits)
            wy = oracle.qwz_dequant(wc, ws, 1, n, B, bits)
            assert_bytes_equal(gather_u16(y, lidx), wy, f"qwZ dequant rank {r} block {b}")
            got_c = gather_bytes(codes, [r * cb + (b * B * bits) // 8], wc.size)
            assert_bytes_equal(got_c, wc, f"qwZ codes rank {r} block {b}")
            assert_f32_bitexact(gather_f32(scales, [r * nb + b]), ws, f"qwZ scale rank {r} block {b}")


def check_qwz(path, wl, nsample=1):
    """Sampled blocks of every rank of a one-call qwZ pass."""
    q = wl.qwz
    assert q.calls == 1
    check_qwz_sampled(path.w_codes[0], path.w_scales[0], path.w_full, q.nranks, q.shard, q.block,
                      q.bits, wl.seed, 0, nsample)


def check_qgz(path, wl, nsample=2):
    g = wl.qgz
    N, G, B, bits = g.nodes, g.gpus_per_node, g.block, g.bits
    Nd, L, bucket = g.nd, g.slice_elems, g.bucket
    blocks = sample_blocks(L // B, nsample, 7)
    nbk = len(blocks)
    Lm = nbk * B
    # mini bucket: rank r, slice j, sampled block q
    pos = (np.arange(Nd)[:, None, None] * L + np.asarray(blocks)[None, :, None] * B
           + np.arange(B)[None, None, :]).reshape(-1)            # slice-relative index j*L + b*B + e
    mbs = []
    for k in range(path.microbatches):
        mini = np.empty(Nd * Nd * Lm, np.uint16)
        for r in range(Nd):
            mini[r * Nd * Lm:(r + 1) * Nd * Lm] = synth.bf16_to_u16(
                synth.at(g.grad, wl.seed, synth.grad_stream(r, k), pos))
        mbs.append(mini)
    if len(mbs) == 1:
        c1, s1 = oracle.qgz_reorder_quant(mbs[0], N, G, Nd * Lm, B, bits)
    else:   # accumulated in arrival order, then quantized from fp32
        acc = oracle.grad_accumulate(mbs)
        c1, s1 = oracle.qgz_reorder_quant_f32(acc, N, G, Nd * Lm, B, bits)
        wa = oracle.grad_accumulate(mbs[:-1])     # what the accumulator holds
        aidx = (np.arange(Nd)[:, None] * bucket + pos[None, :]).reshape(-1)  # rank-major, as wa
        assert_f32_bitexact(gather_f32(path.acc, aidx), wa, "accumulator")
    perm = oracle.qgz_slice_perm(N, G)
    cbr, cbm = oracle.codes_bytes(bucket, bits), oracle.codes_bytes(Nd * Lm, bits)
    bb = B * bits // 8
    # one-shot messages of every rank at every slice position
    starts, wstarts, sidx, widx = [], [], [], []
    for r in range(Nd):
        for p in range(Nd):
            for qi, b in enumerate(blocks):
                starts.append(r * cbr + ((p * L + b * B) * bits) // 8)
                wstarts.append(r * cbm + ((p * Lm + qi * B) * bits) // 8)
                sidx.append(r * (bucket // B) + (p * L + b * B) // B)
                widx.append(r * (Nd * Lm // B) + p * nbk + qi)
    got = gather_bytes(path.msg1, starts, bb)
    want = c1.reshape(-1)[(np.asarray(wstarts)[:, None] + np.arange(bb)[None, :]).reshape(-1)]
    assert_bytes_equal(got, want, "one-shot codes")
    assert_f32_bitexact(gather_f32(path.msg1_scales, sidx), s1[widx], "one-shot scales")
    assert perm is not None
    if N == 1:
        gref = oracle.qgz_hop1(c1, s1, N, G, Nd * Lm, B, bits)
    else:
        c2, s2 = oracle.qgz_hop1(c1, s1, N, G, Nd * Lm, B, bits)
        NL, NLm = N * L, N * Lm
        cb2, cb2m = oracle.codes_bytes(NL, bits), oracle.codes_bytes(NLm, bits)
        starts, wstarts, sidx, widx = [], [], [], []
        for d in range(Nd):
            for k in range(N):
                for qi, b in enumerate(blocks):
                    starts.append(d * cb2 + ((k * L + b * B) * bits) // 8)
                    wstarts.append(d * cb2m + ((k * Lm + qi * B) * bits) // 8)
                    sidx.append(d * (NL // B) + (k * L + b * B) // B)
                    widx.append(d * (NLm // B) + k * nbk + qi)
        got = gather_bytes(path.msg2, starts, bb)
        want = c2.reshape(-1)[(np.asarray(wstarts)[:, None] + np.arange(bb)[None, :]).reshape(-1)]
        assert_bytes_equal(got, want, "hop-1 codes")
        assert_f32_bitexact(gather_f32(path.msg2_scales, sidx), s2[widx], "hop-1 scales")
        gref = oracle.qgz_hop2(c2, s2, N, G, Nd * Lm, B, bits)
    # reduced gradient and Adam state of every rank's sampled blocks
    gidx = (np.arange(Nd)[:, None, None] * L + np.asarray(blocks)[None, :, None] * B
            + np.arange(B)[None, None, :]).reshape(-1)               # global parameter index
    if path.grad_out is not None:
        got_g = gather_f32(path.grad_out, gidx)
        assert_grad_close(got_g, gref, B, "reduced gradient")
        assert_f32_bitexact(got_g, gref, "reduced gradient (bit-exact)")
    if path.adam is not None:
        a = wl.adam
        p0 = oracle.bf16_bits_to_f32(synth.bf16_to_u16(
            synth.at(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, gidx)))
        z = np.zeros(gidx.size, np.float32)
        wp, wm, wv, wb = oracle.adam_step(gref, p0, z, z, a.lr, a.beta1, a.beta2, a.eps, a.step)
        assert_rel_close(gather_f32(path.master, gidx), wp, 1e-5, "master")
        assert_rel_close(gather_f32(path.m, gidx), wm, 1e-5, "m")
        assert_rel_close(gather_f32(path.v, gidx), wv, 1e-5, "v")
        assert_bf16_ulp(gather_u16(path.param, gidx), wb, "param")
        if path.fuse_qwz:   # next step's weight message from the new parameters
            wc, ws = oracle.qwz_quant(wb, Nd, Lm, B, 8)
            got_c = gather_bytes(path.w_codes[0], gidx[::B], B).reshape(-1)
            assert_bytes_equal(got_c, wc, "fused qwZ codes")
            assert_f32_bitexact(gather_f32(path.w_scales[0], gidx[::B] // B), ws,
                                "fused qwZ scales")


@pytest.mark.parametrize("name", ["tiny", "llama", "two_hop", "7b"])
def test_workload_full_size(name):
    """The bench's pass of each workload (the 7B one with its standalone Adam
    shard), every output element against the oracle."""
    Z = zpp()
    wl = W.WORKLOADS[name]
    torch.cuda.empty_cache()
    path = build_path(Z, wl, standalone=True)
    run_checked(path, wl)
    del path
    torch.cuda.empty_cache()


def test_llama_fused_adam_qwz_full_size():
    """The llama step with the weights' qwZ message produced inside the final
    hop's Adam pass (the owned slices are the qwZ shards)."""
    Z = zpp()
    wl = W.WORKLOADS["llama"]
    torch.cuda.empty_cache()
    path = build_path(Z, wl, fuse_qwz=True)
    run_checked(path, wl, fused_prime=True)
    del path
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,microbatches", [("llama", 3), ("two_hop", 2)])
def test_gradient_accumulation_full_size(name, microbatches):
    """Gradient accumulation over micro-batches before the qgZ reduce: the
    accumulator after M-1 micro-batches, the one-shot messages of the
    accumulated bucket, the hops and the fused Adam, every element."""
    Z = zpp()
    wl = W.WORKLOADS[name]
    torch.cuda.empty_cache()
    path = build_path(Z, wl, microbatches=microbatches)
    run_checked(path, wl)
    del path
    torch.cuda.empty_cache()


def test_7b_standalone_adam_full_size():
    """Standalone Adam on the 7B workload's 109,375,000-parameter owned shard
    at step 7 from drawn moments, every element."""
    Z = zpp()
    n = W.SEVEN_B.standalone_adam
    g = synth.fill(W.GRAD_NORMAL, 3, synth.grad_stream(0), 0, n, device="cuda").float()
    master = synth.fill(W.WEIGHT_RECIPE, 3, synth.WEIGHTS, 0, n, device="cuda").float()
    m = synth.fill(W.MOMENT_M_RECIPE, 3, synth.MOMENT_M, 0, n, device="cuda").float()
    v = synth.fill(W.MOMENT_V_RECIPE, 3, synth.MOMENT_V, 0, n, device="cuda").float()
    param = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    hp = (1e-4, 0.9, 0.999, 1e-8, 7)
    Z.zpp_shard_adam_step(g, n, hp, (master, m, v, param))
    torch.cuda.synchronize()
    del g
    F.check_adam_complete((master, m, v, param), n, 3, hp, W.GRAD_NORMAL, synth.grad_stream(0))


def qgz_need_bytes(g):
    c = g.bits / 8 + 4 / g.block
    return g.nd * g.bucket * (2 + c + c / g.gpus_per_node) + 4 * g.bucket


def qwz_need_bytes(q, nranks=None):
    c = q.bits / 8 + 4 / q.block
    return (q.nranks if nranks is None else nranks) * q.shard * (2 + 2 + c)


def run_qwz_rank_groups(Z, q, seed, ranks_per_call):
    """The qwZ half of a sweep point too large for one call's buffers: its
    shards are independent, so they run as calls over groups of ranks (each
    with its weights at the group's global offset), checked on sampled
    blocks of every rank."""
    cb, nb = Z.zpp_codes_bytes(q.shard, q.bits), Z.zpp_num_blocks(q.shard, q.block)
    for r0 in range(0, q.nranks, ranks_per_call):
        n = min(ranks_per_call, q.nranks - r0)
        w = torch.empty(n * q.shard, dtype=torch.bfloat16, device="cuda")
        synth.fill(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, r0 * q.shard, n * q.shard, out=w,
                   chunk=1 << 27)
        codes = torch.empty(n * cb, dtype=torch.uint8, device="cuda")
        scales = torch.empty(n * nb, device="cuda")
        Z.zpp_qwz_quant(w, n, q.shard, q.block, q.bits, codes, scales)
        Z.zpp_qwz_dequant(codes, scales, n, q.shard, q.block, q.bits, w)   # in place: w is y now
        torch.cuda.synchronize()
        check_qwz_sampled(codes, scales, w, n, q.shard, q.block, q.bits, seed, r0 * q.shard)
        del w, codes, scales
        torch.cuda.empty_cache()


@pytest.mark.parametrize("index", range(144))
def test_sweep_point(index):
    """Every sweep point (no Adam): completely where N_d * bucket <= 2^30
    elements, else on sampled blocks of every shard and slice.  A point whose
    buffers do not fit in one pass runs its qgZ chain and its qwZ calls
    separately (the qwZ shards in groups of ranks); only a qgZ chain that does
    not fit by itself is skipped."""
    import dataclasses
    Z = zpp()
    wl = dict(W.sweep_points())[index]
    g, q = wl.qgz, wl.qwz
    torch.cuda.empty_cache()
    budget = 0.85 * torch.cuda.mem_get_info()[0]
    complete = g.nd * g.bucket <= COMPLETE_MAX_ELEMS
    if qgz_need_bytes(g) + qwz_need_bytes(q) <= budget:
        path = build_path(Z, wl, keep_grad=True)
        if complete:
            run_checked(path, wl)
        else:
            path.run()
            torch.cuda.synchronize()
            check_qwz(path, wl, nsample=1)
            check_qgz(path, wl, nsample=1)
        del path
        torch.cuda.empty_cache()
        return
    assert not complete
    if qgz_need_bytes(g) > budget:
        pytest.skip(f"device memory: the qgZ chain needs {qgz_need_bytes(g) / 2**30:.0f} GiB, "
                    f"{budget / 0.85 / 2**30:.0f} GiB free")
    path = build_path(Z, dataclasses.replace(wl, qwz=None), keep_grad=True)
    path.run()
    torch.cuda.synchronize()
    check_qgz(path, wl, nsample=1)
    del path
    torch.cuda.empty_cache()
    budget = 0.85 * torch.cuda.mem_get_info()[0]
    run_qwz_rank_groups(Z, q, wl.seed, max(1, int(budget // qwz_need_bytes(q, 1))))


@pytest.mark.parametrize("nodes", [1, 2, 4])
def test_llama_hpz_backward_gather_full_size(nodes):
    """The llama-layer weights on nodes x (8 / nodes) ranks: the backward
    gather from the secondary partitions rebuilds exactly the weights of the
    forward all-gather."""
    Z = zpp()
    wl = W.WORKLOADS["llama"]
    q = wl.qwz
    qs = Z.QwzSpec(q.nranks, q.shard, q.block, q.bits, nodes=nodes)
    torch.cuda.empty_cache()
    path = Z.CodecPath(qs, None, None, device="cuda", hpz=True)
    synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, qs.phi, out=path.w)
    cap = F.QwzCapture(path, wl)
    path.run_qwz(mark=cap)
    cap.finish()
    fwd = path.w_full.clone()
    path.w_full.zero_()
    path.run_hpz()
    torch.cuda.synchronize()
    assert torch.equal(path.w_full.view(torch.int16), fwd.view(torch.int16))
    del path, fwd
    torch.cuda.empty_cache()


def test_two_hop_bucket_ring_reduce_scatter_full_size():
    """The quantized ring over the two-hop workload's 16 ranks of 2^28-element
    buckets, every reduced-gradient float (blocks restart at chunk starts, so
    the ring over a group of block positions alone reproduces them)."""
    Z = zpp()
    g = W.WORKLOADS["two_hop"].qgz
    nd, bucket, B, bits = g.nd, g.bucket, g.block, g.bits
    L = bucket // nd
    torch.cuda.empty_cache()
    x = grads_for(g, 0, device="cuda")
    cb, nb = Z.zpp_codes_bytes(L, bits), L // B
    bufs = [(torch.empty(nd * cb, dtype=torch.uint8, device="cuda"),
             torch.empty(nd * nb, device="cuda")) for _ in range(2)]
    grad = torch.full((bucket,), float("nan"), device="cuda")
    for step in range(nd):
        ci, si = bufs[(step + 1) & 1] if step else (None, None)
        co, so = bufs[step & 1] if step < nd - 1 else (None, None)
        Z.zpp_ring_rs_step(step, nd, bucket, B, bits, x, ci, si, co, so,
                           grad if step == nd - 1 else None)
    torch.cuda.synchronize()
    del x, bufs
    F.check_ring_complete(grad, g, 0)
    del grad
    torch.cuda.empty_cache()
