"""GPU parity, small cases: the CUDA path through the C ABI against the CPU
oracle, element by element, on seeded inputs that span several warp units and
CTA passes, ragged tails, every supported block size and both bit widths.

Bar: codes, scales and the slice permutation bit-exact; reduced gradients
within 1e-6 of the block's largest magnitude; Adam master/m/v within 1e-5
relative; bf16 parameters within 1 ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W
from gpu_helpers import (assert_bf16_ulp, assert_bytes_equal, assert_f32_bitexact,
                         assert_grad_close, assert_rel_close, np_bytes, np_f32, u16, zpp)

pytestmark = pytest.mark.gpu
BLOCKS = [64, 128, 256, 512, 1024, 2048, 4096]
RNG = np.random.default_rng(7)


def special_values(n, bits, block, rng):
    """fp32 values exercising every quantizer path: plain, all-zero blocks,
    exact ties (x/s = k + 1/2), subnormal scales and single-spike blocks."""
    qmax = (1 << (bits - 1)) - 1
    x = (rng.standard_normal(n) * 0.02).astype(np.float32)
    nb = -(-n // block)
    for b in range(nb):
        lo, hi = b * block, min(n, (b + 1) * block)
        kind = b % 6
        e = 2.0 ** int(rng.integers(-20, 4))
        if kind == 1:
            x[lo:hi] = 0
        elif kind == 2:      # ties: absmax qmax * 2^e, others (k + 1/2) 2^e
            k = rng.integers(-qmax, qmax, size=hi - lo)
            x[lo:hi] = (k + 0.5) * e
            x[lo] = qmax * e
        elif kind == 3:      # subnormal scale
            x[lo:hi] = rng.integers(-1000, 1000, size=hi - lo) * 2.0 ** -142
        elif kind == 4:      # one spike
            x[lo:hi] = 0
            x[lo + int(rng.integers(0, hi - lo))] = -3.0
    return x


def to_dev_bf16(x_f32, dev="cuda"):
    return synth.u16_to_bf16(oracle.f32_to_bf16(x_f32)).to(dev)


# ---- qwZ -------------------------------------------------------------------------------

QWZ_SHAPES = [(1, 1), (1, 7), (1, 1000), (3, 4096), (2, 5000), (4, 3 * 4096 + 64),
              (5, 777), (2, 9 * 1024 + 8), (1, 2 ** 17 + 40), (6, 2 * 4096 + 250)]


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("nranks,shard", QWZ_SHAPES)
def test_qwz_quant_dequant(bits, block, nranks, shard):
    Z = zpp()
    if bits == 4 and shard % 2:
        shard += 1
    n = nranks * shard
    x = special_values(n, bits, block, RNG) if (block + shard) % 3 else \
        (RNG.standard_t(3, n) * 1e-3).astype(np.float32)
    xb = oracle.f32_to_bf16(x)
    want_c, want_s = oracle.qwz_quant(xb, nranks, shard, block, bits)
    want_y = oracle.qwz_dequant(want_c, want_s, nranks, shard, block, bits)

    xd = synth.u16_to_bf16(xb).cuda()
    codes = torch.full((want_c.size,), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((want_s.size,), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    Z.zpp_qwz_quant(xd, nranks, shard, block, bits, codes, scales)
    Z.zpp_qwz_dequant(codes, scales, nranks, shard, block, bits, y)
    torch.cuda.synchronize()
    assert_bytes_equal(np_bytes(codes), want_c, "codes")
    assert_f32_bitexact(np_f32(scales), want_s, "scales")
    assert_bytes_equal(u16(y), want_y, "dequant")


def test_qwz_dequant_of_oracle_codes_and_empty_calls():
    """Dequant alone on codes the oracle wrote; zero-sized calls are no-ops."""
    Z = zpp()
    nranks, shard, block = 3, 5000, 256
    x = oracle.f32_to_bf16((RNG.standard_normal(nranks * shard) * 0.02).astype(np.float32))
    c, s = oracle.qwz_quant(x, nranks, shard, block, 8)
    y = torch.empty(nranks * shard, dtype=torch.bfloat16, device="cuda")
    Z.zpp_qwz_dequant(torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), nranks, shard,
                      block, 8, y)
    torch.cuda.synchronize()
    assert_bytes_equal(u16(y), oracle.qwz_dequant(c, s, nranks, shard, block, 8), "dequant")
    e = torch.empty(0, device="cuda")
    Z.zpp_qwz_quant(e.bfloat16(), 0, 100, 256, 8, e.byte(), e)
    Z.zpp_qwz_quant(e.bfloat16(), 4, 0, 256, 4, e.byte(), e)
    torch.cuda.synchronize()


# ---- qgZ ----------------------------------------------------------------------------------

TOPOS = [(1, 1), (1, 4), (2, 1), (2, 2), (2, 3), (3, 2), (4, 2), (2, 8), (1, 8), (4, 4)]


def qgz_case(N, G, block, bits, slice_blocks, rng, special=False):
    Nd = N * G
    L = slice_blocks * block
    bucket = Nd * L
    if special:
        x = special_values(Nd * bucket, bits, block, rng)
    else:
        x = (rng.standard_t(3, Nd * bucket) * 1e-3).astype(np.float32)
    return Nd, L, bucket, oracle.f32_to_bf16(x)


def run_gpu_chain(Z, gb, N, G, bucket, block, bits, adam=None, state=None, keep_grad=True):
    Nd = N * G
    L = bucket // Nd
    g = synth.u16_to_bf16(gb).cuda()
    c1 = torch.full((Nd * Z.zpp_codes_bytes(bucket, bits),), 0x5A, dtype=torch.uint8, device="cuda")
    s1 = torch.full((Nd * (bucket // block),), float("nan"), device="cuda")
    Z.zpp_qgz_reorder_quant(g, N, G, bucket, block, bits, c1, s1)
    out = {"c1": c1, "s1": s1}
    grad = torch.full((bucket,), float("nan"), device="cuda") if keep_grad else None
    if N == 1:
        Z.zpp_qgz_hop_reduce(1, c1, s1, N, G, bucket, block, bits, grad_out=grad, adam=adam,
                             state=state)
    else:
        nl = N * L
        c2 = torch.full((Nd * Z.zpp_codes_bytes(nl, bits),), 0x5A, dtype=torch.uint8, device="cuda")
        s2 = torch.full((Nd * (nl // block),), float("nan"), device="cuda")
        Z.zpp_qgz_hop_reduce(1, c1, s1, N, G, bucket, block, bits, codes_out=c2, scales_out=s2)
        Z.zpp_qgz_hop_reduce(2, c2, s2, N, G, bucket, block, bits, grad_out=grad, adam=adam,
                             state=state)
        out.update(c2=c2, s2=s2)
    torch.cuda.synchronize()
    out["grad"] = grad
    return out


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block", [64, 256, 1024, 4096])
@pytest.mark.parametrize("N,G", TOPOS)
def test_qgz_chain(bits, block, N, G):
    Z = zpp()
    slice_blocks = {64: 19, 256: 5, 1024: 3, 4096: 1}[block]
    Nd, L, bucket, gb = qgz_case(N, G, block, bits, slice_blocks, RNG, special=(N + G) % 2 == 0)
    c1, s1 = oracle.qgz_reorder_quant(gb, N, G, bucket, block, bits)
    got = run_gpu_chain(Z, gb, N, G, bucket, block, bits)
    assert_bytes_equal(np_bytes(got["c1"]), c1, "one-shot codes")
    assert_f32_bitexact(np_f32(got["s1"]), s1, "one-shot scales")
    if N == 1:
        want = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
    else:
        c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
        assert_bytes_equal(np_bytes(got["c2"]), c2, "hop-1 codes")
        assert_f32_bitexact(np_f32(got["s2"]), s2, "hop-1 scales")
        want = oracle.qgz_hop2(c2, s2, N, G, bucket, block, bits)
    g = np_f32(got["grad"])
    assert_grad_close(g, want, block, "reduced gradient")
    assert_f32_bitexact(g, want, "reduced gradient (bit-exact by construction)")


def hop1_input(N, G, block, bits, L, rng):
    """One-shot messages of Student-t gradients (scales well below 2^-5) with
    outlier, all-zero and subnormal-scale blocks mixed in, so that both int4
    dequantization paths of hop 1 (one FMA a code when every scale of a chunk
    is below 2^-5, the magic-number decode otherwise) run in one launch."""
    Nd = N * G
    bucket = Nd * L
    x = (rng.standard_t(3, Nd * bucket) * 1e-3).astype(np.float32)
    nb = Nd * bucket // block
    xb = x.reshape(nb, block)
    xb[::37] *= 100.0                         # scales above 2^-5
    xb[5::41] = 0.0                           # zero scales
    xb[11::43] = rng.integers(-500, 500, size=xb[11::43].shape) * 2.0 ** -140  # subnormal scales
    c1, s1 = oracle.qgz_reorder_quant(oracle.f32_to_bf16(x), N, G, bucket, block, bits)
    return bucket, c1, s1


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block", [64, 128, 256, 512, 1024, 2048, 4096])
@pytest.mark.parametrize("N,G", [(2, 4), (2, 8), (3, 8)])
def test_hop1_whole_unit_slices(bits, block, N, G):
    """Hop 1 where every destination row is whole 1024-element warp units and
    G is a multiple of four (the per-lane 32-element kernel), against the oracle."""
    Z = zpp()
    L = 2 * max(1024, block)
    bucket, c1, s1 = hop1_input(N, G, block, bits, L, RNG)
    c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
    nl = N * L
    Nd = N * G
    out_c = torch.full((Nd * Z.zpp_codes_bytes(nl, bits),), 0x5A, dtype=torch.uint8, device="cuda")
    out_s = torch.full((Nd * (nl // block),), float("nan"), device="cuda")
    Z.zpp_qgz_hop_reduce(1, torch.from_numpy(c1).cuda(), torch.from_numpy(s1).cuda(), N, G,
                         bucket, block, bits, codes_out=out_c, scales_out=out_s)
    torch.cuda.synchronize()
    assert_bytes_equal(np_bytes(out_c), c2, "hop-1 codes")
    assert_f32_bitexact(np_f32(out_s), s2, "hop-1 scales")


@pytest.mark.parametrize("block", [128, 512, 2048])
def test_hop1_several_units_a_warp(block):
    """Int4 hop 1 with eight sources on a bucket large enough that warp groups
    get more than one unit each (the grid is capped at a few rounds of resident
    CTAs), so stages are refilled and, for B = 2048, the two-slot cross-warp
    absmax alternates; random one-shot messages with scales above 2^-5, zero and
    subnormal scales mixed in, against the oracle."""
    Z = zpp()
    N, G, bits = 2, 8, 4
    Nd = N * G
    L = 1 << 19
    bucket = Nd * L
    rng = np.random.default_rng(block)
    c1 = rng.integers(0, 256, size=Nd * bucket // 2, dtype=np.uint8)
    s1 = (rng.random(Nd * bucket // block, dtype=np.float32) * 1e-3).astype(np.float32)
    s1[::29] *= 100.0                                  # above 2^-5
    s1[3::31] = 0.0
    s1[7::37] = rng.integers(1, 5000, size=s1[7::37].shape) * np.float32(2.0 ** -149)
    c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
    nl = N * L
    out_c = torch.full((Nd * Z.zpp_codes_bytes(nl, bits),), 0x5A, dtype=torch.uint8, device="cuda")
    out_s = torch.full((Nd * (nl // block),), float("nan"), device="cuda")
    Z.zpp_qgz_hop_reduce(1, torch.from_numpy(c1).cuda(), torch.from_numpy(s1).cuda(), N, G,
                         bucket, block, bits, codes_out=out_c, scales_out=out_s)
    torch.cuda.synchronize()
    assert_bytes_equal(np_bytes(out_c), c2, "hop-1 codes")
    assert_f32_bitexact(np_f32(out_s), s2, "hop-1 scales")


def test_slice_permutation_through_the_message():
    """The permutation is read back from the message itself: rank r's slice j,
    filled with a constant that identifies (r, j), must be found at position
    l'*N + n' with j = n'*G + l'."""
    Z = zpp()
    N, G, block, bits = 3, 4, 64, 8
    Nd = N * G
    L, bucket = 2 * block, Nd * 2 * block
    x = np.zeros((Nd, Nd, L), np.float32)
    for r in range(Nd):
        for j in range(Nd):
            x[r, j, :] = r * 16 + j + 1        # <= 188: exact in bf16
            x[r, j, 0] = 1000.0                # same absmax everywhere
    gb = oracle.f32_to_bf16(x.reshape(-1))
    got = run_gpu_chain(Z, gb, N, G, bucket, block, bits)
    q = np_bytes(got["c1"]).view(np.int8).reshape(Nd, Nd, L)
    perm = Z.zpp_qgz_slice_perm(N, G)
    for r in range(Nd):
        for p in range(Nd):
            j = perm[p]
            want = np.rint(np.float32(r * 16 + j + 1) / (np.float32(1000.0) / np.float32(127)))
            assert q[r, p, 1] == want


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,G", [(1, 8), (2, 2), (2, 8), (3, 2)])
def test_final_hop_fused_adam(bits, N, G):
    Z = zpp()
    block = 256
    Nd, L, bucket, gb = qgz_case(N, G, block, bits, 6, RNG)
    want_g = oracle.qgz_reduce_scatter(gb, N, G, bucket, block, bits)
    p0 = (RNG.standard_normal(bucket) * 0.02).astype(np.float32)
    m0 = (RNG.standard_normal(bucket) * 1e-4).astype(np.float32)
    v0 = np.abs(RNG.standard_normal(bucket) * 1e-6).astype(np.float32)
    hp = (1e-4, 0.9, 0.999, 1e-8, 3)
    wp, wm, wv, wb = oracle.adam_step(want_g, p0, m0, v0, *hp)
    master, m, v = (torch.from_numpy(a.copy()).cuda() for a in (p0, m0, v0))
    param = torch.empty(bucket, dtype=torch.bfloat16, device="cuda")
    got = run_gpu_chain(Z, gb, N, G, bucket, block, bits, adam=hp, state=(master, m, v, param))
    assert_f32_bitexact(np_f32(got["grad"]), want_g, "gradient")
    assert_rel_close(np_f32(master), wp, 1e-5, "master")
    assert_rel_close(np_f32(m), wm, 1e-5, "m")
    assert_rel_close(np_f32(v), wv, 1e-5, "v")
    assert_bf16_ulp(u16(param), wb, "param")
    # the kernel evaluates the same IEEE operations in the same order
    assert_f32_bitexact(np_f32(master), wp, "master (bit-exact)")


def test_fused_adam_without_grad_out_and_no_param():
    Z = zpp()
    N, G, block, bits = 2, 4, 512, 4
    Nd, L, bucket, gb = qgz_case(N, G, block, bits, 2, RNG)
    want_g = oracle.qgz_reduce_scatter(gb, N, G, bucket, block, bits)
    z = np.zeros(bucket, np.float32)
    p0 = (RNG.standard_normal(bucket) * 0.02).astype(np.float32)
    wp, wm, wv, _ = oracle.adam_step(want_g, p0, z, z, 1e-4, 0.9, 0.999, 1e-8, 1)
    master = torch.from_numpy(p0.copy()).cuda()
    m = torch.zeros(bucket, device="cuda")
    v = torch.zeros(bucket, device="cuda")
    run_gpu_chain(Z, gb, N, G, bucket, block, bits, adam=(1e-4, 0.9, 0.999, 1e-8, 1),
                  state=(master, m, v, None), keep_grad=False)
    assert_f32_bitexact(np_f32(master), wp, "master")
    assert_f32_bitexact(np_f32(m), wm, "m")
    assert_f32_bitexact(np_f32(v), wv, "v")


@pytest.mark.parametrize("n", [1, 7, 8, 9, 511, 512, 1000, 123457])
@pytest.mark.parametrize("t", [1, 2, 50])
def test_standalone_adam(n, t):
    Z = zpp()
    g = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    p0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    m0 = (RNG.standard_normal(n) * 1e-4).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    v0 = np.abs(RNG.standard_normal(n) * 1e-6).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    hp = (3e-4, 0.9, 0.95, 1e-6, t)
    wp, wm, wv, wb = oracle.adam_step(g, p0, m0, v0, *hp)
    master, m, v = (torch.from_numpy(a.copy()).cuda() for a in (p0, m0, v0))
    param = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    Z.zpp_shard_adam_step(torch.from_numpy(g).cuda(), n, hp, (master, m, v, param))
    torch.cuda.synchronize()
    assert_rel_close(np_f32(master), wp, 1e-5, "master")
    assert_rel_close(np_f32(m), wm, 1e-5, "m")
    assert_rel_close(np_f32(v), wv, 1e-5, "v")
    assert_bf16_ulp(u16(param), wb, "param")
    assert_f32_bitexact(np_f32(master), wp, "master (bit-exact)")


def test_tiny_workload_end_to_end():
    """The tiny workload through CodecPath (the sequence the bench times)."""
    Z = zpp()
    from gradient_comm_codecs_gb300 import AdamSpec, CodecPath, QgzSpec, QwzSpec
    wl = W.TINY
    q, g = wl.qwz, wl.qgz
    path = CodecPath(QwzSpec(q.nranks, q.shard, q.block, q.bits),
                     QgzSpec(g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits),
                     AdamSpec(), device="cuda", keep_grad=True)
    w = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, q.phi)
    path.w.copy_(w)
    from gpu_helpers import grads_for
    grads = grads_for(g, wl.seed)
    path.grads.copy_(grads)
    master0 = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, g.bucket).float()
    path.master.copy_(master0)
    path.run()
    torch.cuda.synchronize()
    wb = u16(w)
    c, s = oracle.qwz_quant(wb, q.nranks, q.shard, q.block, q.bits)
    assert_bytes_equal(u16(path.w_full), oracle.qwz_dequant(c, s, q.nranks, q.shard, q.block,
                                                            q.bits), "qwZ all-gather")
    gref = oracle.qgz_reduce_scatter(u16(grads), g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    assert_f32_bitexact(np_f32(path.grad_out), gref, "reduced gradient")
    z = np.zeros(g.bucket, np.float32)
    wp, wm, wv, wpb = oracle.adam_step(gref, master0.numpy(), z, z, wl.adam.lr, wl.adam.beta1,
                                       wl.adam.beta2, wl.adam.eps, wl.adam.step)
    assert_rel_close(np_f32(path.master), wp, 1e-5, "master")
    assert_bf16_ulp(u16(path.param), wpb, "param")


def test_codec_path_with_standalone_shard_and_microbatches():
    """CodecPath with gradient accumulation over 3 micro-batches and a
    standalone Adam shard (ragged size) after the reduce, two steps."""
    Z = zpp()
    from gradient_comm_codecs_gb300 import AdamSpec, CodecPath, QgzSpec
    from gpu_helpers import grads_for
    wl = W.TINY
    g = wl.qgz
    n_sa = 70001
    path = CodecPath(None, QgzSpec(g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits),
                     AdamSpec(), device="cuda", keep_grad=True, microbatches=3,
                     standalone_adam=n_sa)
    mbs = [grads_for(g, wl.seed, microbatch=k) for k in range(3)]
    for t, mb in zip(path.grads_mb, mbs):
        t.copy_(mb)
    master0 = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, g.bucket).float()
    path.master.copy_(master0)
    sg = (RNG.standard_normal(n_sa) * 1e-3).astype(np.float32)
    sp = (RNG.standard_normal(n_sa) * 0.02).astype(np.float32)
    path.sa_grad.copy_(torch.from_numpy(sg))
    path.sa_master.copy_(torch.from_numpy(sp))
    acc = oracle.grad_accumulate([u16(t) for t in mbs])
    c1, s1 = oracle.qgz_reorder_quant_f32(acc, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    c2, s2 = oracle.qgz_hop1(c1, s1, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    gref = oracle.qgz_hop2(c2, s2, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    a = wl.adam
    p, m, v = master0.numpy(), np.zeros(g.bucket, np.float32), np.zeros(g.bucket, np.float32)
    q, qm, qv = sp, np.zeros(n_sa, np.float32), np.zeros(n_sa, np.float32)
    for step in (1, 2):
        path.run(adam_step=step)
        torch.cuda.synchronize()
        assert_f32_bitexact(np_f32(path.grad_out), gref, f"reduced gradient, step {step}")
        p, m, v, pb = oracle.adam_step(gref, p, m, v, a.lr, a.beta1, a.beta2, a.eps, step)
        q, qm, qv, qb = oracle.adam_step(sg, q, qm, qv, a.lr, a.beta1, a.beta2, a.eps, step)
        assert_f32_bitexact(np_f32(path.master), p, f"master, step {step}")
        assert_bf16_ulp(u16(path.param), pb, f"param, step {step}")
        assert_f32_bitexact(np_f32(path.sa_master), q, f"standalone master, step {step}")
        assert_f32_bitexact(np_f32(path.sa_v), qv, f"standalone v, step {step}")
        assert_bf16_ulp(u16(path.sa_param), qb, f"standalone param, step {step}")


# ---- next row: Adam -> qwZ of the new parameters, fused into the final hop -----------------------

@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,G,block", [(1, 8, 512), (2, 2, 256), (2, 4, 1024), (4, 2, 2048),
                                       (1, 4, 64), (2, 2, 4096)])
def test_final_hop_adam_qwz(bits, N, G, block):
    Z = zpp()
    Nd = N * G
    L = 3 * max(block, 512)
    bucket = Nd * L
    x = (RNG.standard_t(3, Nd * bucket) * 1e-3).astype(np.float32)
    gb = oracle.f32_to_bf16(x)
    c1, s1 = oracle.qgz_reorder_quant(gb, N, G, bucket, block, bits)
    if N == 1:
        gref = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
        hop, ci, si = 1, torch.from_numpy(c1).cuda(), torch.from_numpy(s1).cuda()
    else:
        c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
        gref = oracle.qgz_hop2(c2, s2, N, G, bucket, block, bits)
        hop, ci, si = 2, torch.from_numpy(c2).cuda(), torch.from_numpy(s2).cuda()
    p0 = (RNG.standard_normal(bucket) * 0.02).astype(np.float32)
    m0 = (RNG.standard_normal(bucket) * 1e-4).astype(np.float32)
    v0 = np.abs(RNG.standard_normal(bucket) * 1e-6).astype(np.float32)
    hp = (1e-4, 0.9, 0.999, 1e-8, 4)
    wp, wm, wv, wb, wc, ws = oracle.adam_then_qwz(gref, p0, m0, v0, *hp, Nd, L, block, 8)
    master, m, v = (torch.from_numpy(a.copy()).cuda() for a in (p0, m0, v0))
    param = torch.empty(bucket, dtype=torch.bfloat16, device="cuda")
    grad = torch.full((bucket,), float("nan"), device="cuda")
    qc = torch.full((bucket,), 0x5A, dtype=torch.uint8, device="cuda")
    qs = torch.full((bucket // block,), float("nan"), device="cuda")
    Z.zpp_qgz_final_hop_adam_qwz(hop, ci, si, N, G, bucket, block, bits, grad, hp,
                                 (master, m, v, param), 8, qc, qs)
    torch.cuda.synchronize()
    assert_f32_bitexact(np_f32(grad), gref, "gradient")
    assert_rel_close(np_f32(master), wp, 1e-5, "master")
    assert_rel_close(np_f32(m), wm, 1e-5, "m")
    assert_rel_close(np_f32(v), wv, 1e-5, "v")
    assert_bf16_ulp(u16(param), wb, "param")
    assert_bytes_equal(np_bytes(qc), wc, "fused qwZ codes")
    assert_f32_bitexact(np_f32(qs), ws, "fused qwZ scales")


def test_final_hop_adam_qwz_rejects_unsupported():
    Z = zpp()
    N, G, block, bits = 1, 4, 256, 4
    bucket = 4 * 768                        # L = 768: not a multiple of 512
    t = torch.zeros(bucket, device="cuda")
    c = torch.zeros(4 * bucket, dtype=torch.uint8, device="cuda")
    st = (t, t.clone(), t.clone(), None)
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_qgz_final_hop_adam_qwz(1, c, t, N, G, bucket, block, bits, None,
                                     (1e-4, 0.9, 0.999, 1e-8, 1), st, 8, c, t)
    assert e.value.status == Z.ZPP_ERR_UNSUPPORTED
    bucket = 4 * 1024
    t = torch.zeros(bucket, device="cuda")
    c = torch.zeros(4 * bucket, dtype=torch.uint8, device="cuda")
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_qgz_final_hop_adam_qwz(1, c, t, N, G, bucket, block, bits, None,
                                     (1e-4, 0.9, 0.999, 1e-8, 1), (t, t.clone(), t.clone(), None),
                                     4, c, t)
    assert e.value.status == Z.ZPP_ERR_UNSUPPORTED


# ---- next row: gradient accumulation before the qgZ reduce --------------------------------------

@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 2047, 123457])
@pytest.mark.parametrize("M", [1, 2, 5])
def test_grad_accumulate(n, M):
    Z = zpp()
    mbs = [oracle.f32_to_bf16((RNG.standard_t(3, n) * 1e-3).astype(np.float32)) for _ in range(M)]
    acc = torch.full((max(n, 1),), float("nan"), device="cuda")[:n]
    for k, g in enumerate(mbs):
        Z.zpp_grad_accumulate(synth.u16_to_bf16(g).cuda(), acc, n, k == 0)
    torch.cuda.synchronize()
    if n:
        assert_f32_bitexact(np_f32(acc), oracle.grad_accumulate(mbs), "accumulator")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block,slice_blocks", [(64, 19), (64, 16), (256, 5), (256, 8),
                                                (1024, 3), (2048, 2), (4096, 1)])
@pytest.mark.parametrize("N,G", [(1, 1), (1, 8), (2, 2), (2, 3), (4, 2)])
@pytest.mark.parametrize("M", [2, 4])
def test_qgz_reorder_quant_acc(bits, block, slice_blocks, N, G, M):
    """One-shot messages of an accumulated bucket: the first M-1 micro-batches
    through zpp_grad_accumulate, the last added inside the quantizer; then the
    hops and the reduced gradient."""
    Z = zpp()
    Nd = N * G
    bucket = Nd * slice_blocks * block
    mbs = [oracle.f32_to_bf16((RNG.standard_t(3, Nd * bucket) * 1e-3).astype(np.float32))
           for _ in range(M)]
    if (N + G + M) % 2 == 0:    # the accumulated bucket exercises the quantizer's special cases
        mbs[0] = oracle.f32_to_bf16(special_values(Nd * bucket, bits, block, RNG))
        for k in range(1, M):
            mbs[k] = np.zeros_like(mbs[0])
    acc_ref = oracle.grad_accumulate(mbs)
    c1, s1 = oracle.qgz_reorder_quant_f32(acc_ref, N, G, bucket, block, bits)
    acc = torch.full((Nd * bucket,), float("nan"), device="cuda")
    for k in range(M - 1):
        Z.zpp_grad_accumulate(synth.u16_to_bf16(mbs[k]).cuda(), acc, Nd * bucket, k == 0)
    torch.cuda.synchronize()
    acc_before = acc.clone()
    codes = torch.full((Nd * Z.zpp_codes_bytes(bucket, bits),), 0x5A, dtype=torch.uint8,
                       device="cuda")
    scales = torch.full((Nd * (bucket // block),), float("nan"), device="cuda")
    Z.zpp_qgz_reorder_quant_acc(synth.u16_to_bf16(mbs[-1]).cuda(), acc, N, G, bucket, block, bits,
                                codes, scales)
    torch.cuda.synchronize()
    assert torch.equal(acc.view(torch.int32), acc_before.view(torch.int32)), "acc was written"
    assert_f32_bitexact(np_f32(acc), oracle.grad_accumulate(mbs[:-1]), "accumulator")
    assert_bytes_equal(np_bytes(codes), c1, "one-shot codes of the accumulated bucket")
    assert_f32_bitexact(np_f32(scales), s1, "one-shot scales of the accumulated bucket")
    grad = torch.full((bucket,), float("nan"), device="cuda")
    if N == 1:
        Z.zpp_qgz_hop_reduce(1, codes, scales, N, G, bucket, block, bits, grad_out=grad)
        want = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
    else:
        nl = bucket // G
        c2 = torch.empty((Nd * Z.zpp_codes_bytes(nl, bits),), dtype=torch.uint8, device="cuda")
        s2 = torch.empty((Nd * (nl // block),), device="cuda")
        Z.zpp_qgz_hop_reduce(1, codes, scales, N, G, bucket, block, bits, codes_out=c2,
                             scales_out=s2)
        Z.zpp_qgz_hop_reduce(2, c2, s2, N, G, bucket, block, bits, grad_out=grad)
        want = oracle.qgz_hop2(*oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits), N, G, bucket,
                               block, bits)
    torch.cuda.synchronize()
    assert_f32_bitexact(np_f32(grad), want, "reduced gradient of the accumulated bucket")


def test_accumulation_arguments():
    Z = zpp()
    g = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    acc = torch.zeros(129, device="cuda")
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_grad_accumulate(g, acc, 64, 2)
    assert e.value.status == Z.ZPP_ERR_INVALID_ARG
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_grad_accumulate(g, acc[1:], 64, 1)
    assert e.value.status == Z.ZPP_ERR_MISALIGNED
    c = torch.zeros(128, dtype=torch.uint8, device="cuda")
    with pytest.raises(Z.ZppError) as e:   # bucket not a multiple of N_d * block
        Z.zpp_qgz_reorder_quant_acc(g, acc, 1, 2, 64, 64, 8, c, acc)
    assert e.value.status == Z.ZPP_ERR_INVALID_ARG
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_qgz_reorder_quant_acc(g, acc[1:], 1, 1, 64, 64, 8, c, acc)
    assert e.value.status == Z.ZPP_ERR_MISALIGNED


# ---- fp32 arrays 16-byte but not 32-byte aligned (the two-128-bit access path) ------------------

def _off16(a: np.ndarray) -> torch.Tensor:
    """A device view of `a` starting 16 bytes into a fresh allocation."""
    buf = torch.empty(a.size + 4, dtype=torch.float32, device="cuda")
    buf[4:].copy_(torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)))
    v = buf[4:]
    assert v.data_ptr() % 32 == 16
    return v


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,G", [(1, 4), (2, 2)])
def test_sixteen_byte_aligned_state(bits, N, G):
    Z = zpp()
    block = 256
    Nd, L, bucket, gb = qgz_case(N, G, block, bits, 6, RNG)
    want_g = oracle.qgz_reduce_scatter(gb, N, G, bucket, block, bits)
    p0 = (RNG.standard_normal(bucket) * 0.02).astype(np.float32)
    m0 = (RNG.standard_normal(bucket) * 1e-4).astype(np.float32)
    v0 = np.abs(RNG.standard_normal(bucket) * 1e-6).astype(np.float32)
    hp = (1e-4, 0.9, 0.999, 1e-8, 3)
    wp, wm, wv, wb = oracle.adam_step(want_g, p0, m0, v0, *hp)
    master, m, v = _off16(p0), _off16(m0), _off16(v0)
    param = torch.empty(bucket, dtype=torch.bfloat16, device="cuda")
    grad = _off16(np.full(bucket, np.nan, np.float32))
    g = synth.u16_to_bf16(gb).cuda()
    c1 = torch.empty(Nd * Z.zpp_codes_bytes(bucket, bits), dtype=torch.uint8, device="cuda")
    s1 = torch.empty(Nd * (bucket // block), device="cuda")
    Z.zpp_qgz_reorder_quant(g, N, G, bucket, block, bits, c1, s1)
    if N == 1:
        Z.zpp_qgz_hop_reduce(1, c1, s1, N, G, bucket, block, bits, grad_out=grad, adam=hp,
                             state=(master, m, v, param))
    else:
        nl = N * L
        c2 = torch.empty(Nd * Z.zpp_codes_bytes(nl, bits), dtype=torch.uint8, device="cuda")
        s2 = torch.empty(Nd * (nl // block), device="cuda")
        Z.zpp_qgz_hop_reduce(1, c1, s1, N, G, bucket, block, bits, codes_out=c2, scales_out=s2)
        Z.zpp_qgz_hop_reduce(2, c2, s2, N, G, bucket, block, bits, grad_out=grad, adam=hp,
                             state=(master, m, v, param))
    torch.cuda.synchronize()
    assert_f32_bitexact(np_f32(grad), want_g, "gradient")
    assert_f32_bitexact(np_f32(master), wp, "master")
    assert_f32_bitexact(np_f32(m), wm, "m")
    assert_f32_bitexact(np_f32(v), wv, "v")
    assert_bf16_ulp(u16(param), wb, "param")
    # standalone Adam and accumulation on the same offset views
    n = bucket - 3
    gs = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    wp2, wm2, wv2, _ = oracle.adam_step(gs, wp[:n], wm[:n], wv[:n], *hp)
    Z.zpp_shard_adam_step(_off16(gs), n, hp, (master, m, v, None))
    torch.cuda.synchronize()
    assert_f32_bitexact(np_f32(master)[:n], wp2, "standalone master")
    assert_f32_bitexact(np_f32(m)[:n], wm2, "standalone m")
    assert_f32_bitexact(np_f32(v)[:n], wv2, "standalone v")
    mbs = [gb[:n], gb[n:2 * n]]
    acc = _off16(np.zeros(n, np.float32))
    for k, mb in enumerate(mbs):
        Z.zpp_grad_accumulate(synth.u16_to_bf16(mb).cuda(), acc, n, k == 0)
    torch.cuda.synchronize()
    assert_f32_bitexact(np_f32(acc), oracle.grad_accumulate(mbs), "accumulator")


# ---- next row: hpZ node-local backward gather from secondary partitions -------------------------

def _hpz_case(N, G, shard, block, bits, rng):
    """Forward qwZ messages of N_d shards and the G secondary partitions kept
    from them, each a separate device allocation."""
    Nd = N * G
    w = oracle.f32_to_bf16((rng.standard_normal(Nd * shard) * 0.02).astype(np.float32))
    if bits == 16:
        secs = [w[l * N * shard:(l + 1) * N * shard].copy() for l in range(G)]
        dev = [synth.u16_to_bf16(s).cuda() for s in secs]
        return w, secs, dev, None
    c, s = oracle.qwz_quant(w, Nd, shard, block, bits)
    cb, nb = oracle.codes_bytes(shard, bits), oracle.num_blocks(shard, block)
    secs = [(c[l * N * cb:(l + 1) * N * cb].copy(), s[l * N * nb:(l + 1) * N * nb].copy())
            for l in range(G)]
    return (c, s), secs, [torch.from_numpy(a).cuda() for a, _ in secs], \
        [torch.from_numpy(b).cuda() for _, b in secs]


@pytest.mark.parametrize("bits", [16, 8, 4])
@pytest.mark.parametrize("shard,block", [(4096, 256), (3 * 1024 + 64, 64), (2 * 4096, 2048),
                                         (1000, 128), (514, 512), (2, 64)])
@pytest.mark.parametrize("N,G", [(1, 8), (2, 4), (4, 2), (3, 3), (2, 8), (1, 1)])
def test_hpz_gather(bits, shard, block, N, G):
    Z = zpp()
    fwd, secs, dc, ds = _hpz_case(N, G, shard, block, bits, RNG)
    want = oracle.hpz_gather(secs, N, shard, block, bits)
    y = torch.full((N * G * shard,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    Z.zpp_hpz_gather(G, N, shard, block, bits, dc, ds, y)
    torch.cuda.synchronize()
    assert_bytes_equal(u16(y), want, "hpZ backward gather")
    if bits != 16:   # the same weights the forward all-gather delivered
        c, s = fwd
        yf = torch.empty_like(y)
        Z.zpp_qwz_dequant(torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), N * G, shard,
                          block, bits, yf)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), yf.view(torch.int16))


def test_hpz_arguments():
    import ctypes
    Z = zpp()
    c = [torch.zeros(4096, dtype=torch.uint8, device="cuda") for _ in range(2)]
    s = [torch.zeros(64, device="cuda") for _ in range(2)]
    y = torch.zeros(2 * 4096, dtype=torch.bfloat16, device="cuda")
    Z.zpp_hpz_gather(2, 1, 4096, 64, 8, c, s, y)
    lib = Z._lib._lib()
    cp = (ctypes.c_void_p * 65)(*([c[0].data_ptr()] * 65))
    sp = (ctypes.c_void_p * 65)(*([s[0].data_ptr()] * 65))
    P = lambda a: ctypes.cast(a, ctypes.c_void_p)   # noqa: E731
    for args in ((65, 1, 4096, 64, 8), (0, 1, 4096, 64, 8), (2, 0, 4096, 64, 8),
                 (2, 1, 4096, 48, 8), (2, 1, 4095, 64, 4), (2, 1, 4096, 64, 2)):
        assert lib.zpp_hpz_gather(*args, P(cp), P(sp), y.data_ptr(), None) == \
            Z.ZPP_ERR_INVALID_ARG, args
    assert lib.zpp_hpz_gather(2, 1, 4096, 64, 8, P(cp), None, y.data_ptr(), None) == \
        Z.ZPP_ERR_INVALID_ARG
    cm = torch.zeros(4096 + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_hpz_gather(2, 1, 4096, 64, 8, [c[0], cm[4:4100]], s, y)
    assert e.value.status == Z.ZPP_ERR_MISALIGNED
    assert Z.zpp_hpz_secondary_bytes(2, 4096, 256, 8) == oracle.hpz_secondary_bytes(2, 4096, 256, 8)
    assert Z.zpp_hpz_secondary_bytes(2, 4096, 256, 16) == 2 * 2 * 4096
    assert Z.zpp_hpz_secondary_bytes(0, 4096, 256, 8) == -1


# ---- next row: quantized ring reduce-scatter (the comparator of qgZ's one-shot scheme) ----------

def run_gpu_ring(Z, gb, nd, bucket, block, bits):
    """Every step on the GPU; returns the messages of each step and the gradient."""
    L = bucket // nd
    x = synth.u16_to_bf16(gb).cuda()
    cb, nb = Z.zpp_codes_bytes(L, bits), L // block
    bufs = [(torch.full((nd * cb,), 0x5A, dtype=torch.uint8, device="cuda"),
             torch.full((nd * nb,), float("nan"), device="cuda")) for _ in range(2)]
    grad = torch.full((bucket,), float("nan"), device="cuda")
    msgs = []
    for step in range(nd):
        ci, si = bufs[(step + 1) & 1] if step else (None, None)
        co, so = bufs[step & 1] if step < nd - 1 else (None, None)
        Z.zpp_ring_rs_step(step, nd, bucket, block, bits, x, ci, si, co, so,
                           grad if step == nd - 1 else None)
        if step < nd - 1:
            torch.cuda.synchronize()
            msgs.append((np_bytes(co).copy(), np_f32(so).copy()))
    torch.cuda.synchronize()
    return msgs, np_f32(grad)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block,chunk_blocks", [(64, 3), (64, 16), (256, 5), (1024, 2),
                                                (4096, 1)])
@pytest.mark.parametrize("nd", [1, 2, 3, 4, 8, 16])
def test_ring_reduce_scatter(bits, block, chunk_blocks, nd):
    Z = zpp()
    L = chunk_blocks * block
    bucket = nd * L
    if (nd + chunk_blocks) % 2:
        x = special_values(nd * bucket, bits, block, RNG)
    else:
        x = (RNG.standard_t(3, nd * bucket) * 1e-3).astype(np.float32)
    gb = oracle.f32_to_bf16(x)
    msgs, g = run_gpu_ring(Z, gb, nd, bucket, block, bits)
    ci = si = None
    for step in range(nd - 1):
        c, s = oracle.ring_rs_step(step, nd, bucket, block, bits, gb, ci, si)
        assert_bytes_equal(msgs[step][0], c, f"ring step {step} codes")
        assert_f32_bitexact(msgs[step][1], s, f"ring step {step} scales")
        ci, si = c, s
    want = oracle.ring_rs_step(nd - 1, nd, bucket, block, bits, gb, ci, si)
    assert_f32_bitexact(g, want, "ring gradient")
    assert_f32_bitexact(g, oracle.ring_reduce_scatter(gb, nd, bucket, block, bits),
                        "ring gradient (whole ring)")


def test_ring_arguments():
    Z = zpp()
    x = torch.zeros(4 * 1024, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    s = torch.zeros(16, device="cuda")
    g = torch.zeros(4 * 256, device="cuda")
    Z.zpp_ring_rs_step(0, 2, 512, 64, 8, x, None, None, c, s)
    for bad in ((2, 2), (-1, 2)):
        with pytest.raises(Z.ZppError) as e:
            Z.zpp_ring_rs_step(bad[0], bad[1], 512, 64, 8, x, c, s, c, s, g)
        assert e.value.status == Z.ZPP_ERR_INVALID_ARG
    with pytest.raises(Z.ZppError) as e:       # a middle step needs its input
        Z.zpp_ring_rs_step(1, 4, 1024, 64, 8, x, None, None, c, s)
    assert e.value.status == Z.ZPP_ERR_INVALID_ARG
    with pytest.raises(Z.ZppError) as e:       # the last step writes the gradient
        Z.zpp_ring_rs_step(1, 2, 512, 64, 8, x, c, s, None, None, None)
    assert e.value.status == Z.ZPP_ERR_INVALID_ARG
    with pytest.raises(Z.ZppError) as e:
        Z.zpp_ring_rs_step(1, 2, 512, 64, 8, x, c, s, None, None, g[1:])
    assert e.value.status == Z.ZPP_ERR_MISALIGNED


# ---- the end-to-end call on host buffers ---------------------------------------------------------

@pytest.mark.parametrize("copy_streams", [1, 3])
def test_run_from_host(copy_streams):
    """CodecPath.run_from_host (chunked copies over several streams overlapping
    the kernels): the parameters copied back are the oracle's, with
    micro-batches, hpZ and a standalone shard in the pass."""
    Z = zpp()
    from gradient_comm_codecs_gb300 import AdamSpec, CodecPath, QgzSpec, QwzSpec
    from gpu_helpers import grads_for
    wl = W.TINY
    q, g = wl.qwz, wl.qgz
    n_sa = 50001
    path = CodecPath(QwzSpec(q.nranks, q.shard, q.block, q.bits, nodes=g.nodes),
                     QgzSpec(g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits), AdamSpec(),
                     device="cuda", keep_grad=True, microbatches=2, standalone_adam=n_sa, hpz=True)
    w = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, q.phi).pin_memory()
    mbs = [grads_for(g, wl.seed, microbatch=k).pin_memory() for k in range(2)]
    master0 = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, g.bucket).float()
    path.master.copy_(master0)
    sg = torch.from_numpy((RNG.standard_normal(n_sa) * 1e-3).astype(np.float32)).pin_memory()
    sp = (RNG.standard_normal(n_sa) * 0.02).astype(np.float32)
    path.sa_master.copy_(torch.from_numpy(sp))
    p_host = torch.empty(g.bucket, dtype=torch.bfloat16).pin_memory()
    sa_host = torch.empty(n_sa, dtype=torch.bfloat16).pin_memory()
    h2d, d2h = path.run_from_host(w, mbs, p_host, adam_step=1, sa_grad_host=sg,
                                  sa_param_host=sa_host, copy_streams=copy_streams)
    torch.cuda.synchronize()
    assert h2d == 2 * q.phi + 2 * 2 * g.nd * g.bucket + 4 * n_sa
    assert d2h == 2 * g.bucket + 2 * n_sa
    c, s = oracle.qwz_quant(u16(w), q.nranks, q.shard, q.block, q.bits)
    assert_bytes_equal(u16(path.w_full), oracle.qwz_dequant(c, s, q.nranks, q.shard, q.block,
                                                            q.bits), "weights gathered (hpZ)")
    acc = oracle.grad_accumulate([u16(t) for t in mbs])
    c1, s1 = oracle.qgz_reorder_quant_f32(acc, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    c2, s2 = oracle.qgz_hop1(c1, s1, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    gref = oracle.qgz_hop2(c2, s2, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
    a = wl.adam
    z = np.zeros(g.bucket, np.float32)
    _, _, _, pb = oracle.adam_step(gref, master0.numpy(), z, z, a.lr, a.beta1, a.beta2, a.eps, 1)
    assert_bf16_ulp(u16(p_host), pb, "parameters copied back")
    zs = np.zeros(n_sa, np.float32)
    _, _, _, qb = oracle.adam_step(sg.numpy(), sp, zs, zs, a.lr, a.beta1, a.beta2, a.eps, 1)
    assert_bf16_ulp(u16(sa_host), qb, "standalone parameters copied back")


@pytest.mark.parametrize("input_sets", [1, 2, 3])
def test_run_from_host_successive_steps(input_sets):
    """Three run_from_host calls in a row with different weights and gradients
    each, over 1-3 sets of device input buffers (the next call's copies in
    flight under this call's kernels): after the third call the gathered
    weights, the reduced gradient and the parameters copied back are the
    oracle's for the third step, with m and v carried over three Adam steps."""
    Z = zpp()
    from gradient_comm_codecs_gb300 import AdamSpec, CodecPath, QgzSpec, QwzSpec
    from gpu_helpers import grads_for
    wl = W.TINY
    q, g = wl.qwz, wl.qgz
    a = wl.adam
    path = CodecPath(QwzSpec(q.nranks, q.shard, q.block, q.bits),
                     QgzSpec(g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits), AdamSpec(),
                     device="cuda", keep_grad=True)
    master0 = synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, g.bucket).float()
    path.master.copy_(master0)
    ws = [synth.fill(W.WEIGHT_RECIPE, 10 + k, synth.WEIGHTS, 0, q.phi).pin_memory()
          for k in range(3)]
    gs = [grads_for(g, wl.seed, microbatch=k).pin_memory() for k in range(3)]
    p_host = torch.empty(g.bucket, dtype=torch.bfloat16).pin_memory()
    for k in range(3):
        path.run_from_host(ws[k], gs[k], p_host, adam_step=1 + k, input_sets=input_sets)
    torch.cuda.synchronize()
    c, s = oracle.qwz_quant(u16(ws[2]), q.nranks, q.shard, q.block, q.bits)
    assert_bytes_equal(u16(path.w_full), oracle.qwz_dequant(c, s, q.nranks, q.shard, q.block,
                                                            q.bits), "third step's weights")
    p, m, v = master0.numpy(), np.zeros(g.bucket, np.float32), np.zeros(g.bucket, np.float32)
    for k in range(3):
        c1, s1 = oracle.qgz_reorder_quant(u16(gs[k]), g.nodes, g.gpus_per_node, g.bucket,
                                          g.block, g.bits)
        c2, s2 = oracle.qgz_hop1(c1, s1, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
        gref = oracle.qgz_hop2(c2, s2, g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits)
        p, m, v, pb = oracle.adam_step(gref, p, m, v, a.lr, a.beta1, a.beta2, a.eps, 1 + k)
    assert_f32_bitexact(np_f32(path.grad_out), gref, "third step's reduced gradient")
    assert_rel_close(np_f32(path.master), p, 1e-5, "master after three steps")
    assert_bf16_ulp(u16(p_host), pb, "parameters copied back after three steps")


def _fuzz_cases(n, seed):
    """Seeded random topologies, block sizes, widths and slice lengths: whole 1024-element
    units or ragged, G a multiple of 4 or not, blocks within or across warps."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        N = int(rng.choice([1, 2, 2, 3, 4]))
        G = int(rng.choice([1, 2, 3, 4, 4, 5, 8, 8, 12, 16]))
        block = int(rng.choice(BLOCKS))
        bits = int(rng.choice([4, 8]))
        if rng.random() < 0.5:  # whole units: L a multiple of max(1024, B)
            L = max(1024, block) * int(rng.integers(1, 4))
        else:
            L = block * int(rng.integers(1, 12))
        Nd = N * G
        if Nd * Nd * L > (1 << 23):
            continue
        cases.append((N, G, block, bits, L, int(rng.integers(0, 1 << 30))))
    return cases


@pytest.mark.parametrize("N,G,block,bits,L,seed", _fuzz_cases(48, 2024))
def test_fuzz_qgz_chain_and_ring(N, G, block, bits, L, seed):
    """Random shapes through every dispatch branch of the reduce: one-shot reorder+quant,
    hop 1, hop 2 (or the single final hop) and the quantized ring, against the oracle."""
    Z = zpp()
    rng = np.random.default_rng(seed)
    Nd = N * G
    bucket = Nd * L
    x = (rng.standard_t(3, Nd * bucket) * 1e-3).astype(np.float32)
    xb = x.reshape(-1, block)
    xb[rng.integers(0, xb.shape[0], size=max(1, xb.shape[0] // 50))] *= 100.0
    gb = oracle.f32_to_bf16(x)
    got = run_gpu_chain(Z, gb, N, G, bucket, block, bits)
    c1, s1 = oracle.qgz_reorder_quant(gb, N, G, bucket, block, bits)
    assert_bytes_equal(np_bytes(got["c1"]), c1, "one-shot codes")
    assert_f32_bitexact(np_f32(got["s1"]), s1, "one-shot scales")
    if N == 1:
        want = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
    else:
        c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket, block, bits)
        assert_bytes_equal(np_bytes(got["c2"]), c2, "hop-1 codes")
        assert_f32_bitexact(np_f32(got["s2"]), s2, "hop-1 scales")
        want = oracle.qgz_hop2(c2, s2, N, G, bucket, block, bits)
    assert_f32_bitexact(np_f32(got["grad"]), want, "reduced gradient")
    _, g = run_gpu_ring(Z, gb, Nd, bucket, block, bits)
    assert_f32_bitexact(g, oracle.ring_reduce_scatter(gb, Nd, bucket, block, bits), "ring")
