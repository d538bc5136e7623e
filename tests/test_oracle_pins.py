"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's formula: each checks it against a hand
worked value, a brute-force search, a closed form, an invariant or an
independent library routine, chosen so that a dropped term, a wrong sign, a
wrong index or a transposed operand fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import accounting
from conftest import golden, golden_rows

RNG = np.random.default_rng(1234)


def f32(x):
    return np.float32(x)


# ---- O1: block quantization -----------------------------------------------------

def brute_force_codes(x, s, qmax):
    """argmin over integers q in [-qmax, qmax] of |fl32(x/s) - q|, ties to even."""
    out = []
    for xi in np.asarray(x, dtype=np.float32):
        if s == 0:
            out.append(0)
            continue
        y = float(np.float32(xi) / np.float32(s))     # IEEE fp32 divide
        best, bestd = None, None
        for q in range(-qmax, qmax + 1):
            d = abs(y - q)
            if bestd is None or d < bestd or (d == bestd and q % 2 == 0):
                best, bestd = q, d
        out.append(best)
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("block", [1, 3, 8, 64])
def test_codes_brute_force(bits, block):
    qmax = (1 << (bits - 1)) - 1
    for trial in range(30):
        n = int(RNG.integers(1, 3 * block + 2))
        scale = float(10.0 ** RNG.uniform(-6, 2))
        x = (RNG.standard_normal(n) * scale).astype(np.float32)
        if trial % 3 == 0:            # bf16-valued inputs, as the path sees them
            x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
        codes, scales = oracle.block_quant(x, block, bits)
        q = oracle.unpack_codes(codes, n, bits)
        for b in range(scales.size):
            blk = x[b * block:(b + 1) * block]
            amax = float(np.max(np.abs(blk)))
            # scale: correctly rounded fp32 of absmax/qmax (double then round
            # is correct rounding for a quotient of fp32 values)
            assert scales[b] == np.float32(amax / qmax)
            assert np.array_equal(q[b * block:(b + 1) * block],
                                  brute_force_codes(blk, scales[b], qmax))


def test_round_half_even_ties_worked_by_hand():
    rows = golden_rows("quant_ties.txt")
    x = np.array([float(r[0]) for r in rows], dtype=np.float32)
    want = np.array([int(r[1]) for r in rows])
    codes, scales = oracle.block_quant(x, x.size, 8)
    assert scales[0] == 1.0
    assert np.array_equal(oracle.unpack_codes(codes, x.size, 8), want)


def test_int4_packing_worked_by_hand():
    x = np.array([7, -7, 1, -1, 0, 3, -4, 5], dtype=np.float32)
    codes, scales = oracle.block_quant(x, 8, 4)
    assert scales[0] == 1.0
    want = {int(r[0]): int(r[1], 16) for r in golden_rows("int4_packing.txt")}
    assert [int(b) for b in codes] == [want[i] for i in range(4)]


@pytest.mark.parametrize("bits", [8, 4])
def test_dequant_error_within_half_scale(bits):
    qmax = (1 << (bits - 1)) - 1
    u = 2.0 ** -24
    for _ in range(20):
        n, block = 4096, int(RNG.choice([64, 256, 1000]))
        x = (RNG.standard_t(3, n) * 1e-3).astype(np.float32)
        codes, scales = oracle.block_quant(x, block, bits)
        y = oracle.block_dequant(codes, scales, n, block, bits).astype(np.float64)
        s = np.repeat(scales.astype(np.float64), block)[:n]
        # |fl(q s) - x| <= s/2 + u(|x| + |q s|) <= s/2 + 2u (qmax+1) s
        bound = s / 2 + 2 * u * (qmax + 1) * s
        assert np.all(np.abs(y - x.astype(np.float64)) <= bound)


@pytest.mark.parametrize("bits", [8, 4])
def test_special_blocks(bits):
    qmax = (1 << (bits - 1)) - 1
    # absmax element -> +-qmax
    x = np.array([0.1, -0.3, 0.25, 0.05], dtype=np.float32)
    c, s = oracle.block_quant(x, 4, bits)
    assert oracle.unpack_codes(c, 4, bits)[1] == -qmax
    # zero block -> scale 0, codes 0
    c, s = oracle.block_quant(np.zeros(6, np.float32), 6, bits)
    assert s[0] == 0 and not oracle.unpack_codes(c, 6, bits).any()
    # one nonzero value -> +-qmax, the rest 0
    x = np.zeros(8, np.float32)
    x[5] = -3e-7
    c, s = oracle.block_quant(x, 8, bits)
    q = oracle.unpack_codes(c, 8, bits)
    assert q[5] == -qmax and np.count_nonzero(q) == 1
    # tail block: scale over the remaining elements only
    x = np.concatenate([np.full(8, 100.0, np.float32), np.array([1.0, -2.0], np.float32)])
    c, s = oracle.block_quant(x, 8, bits)
    assert s.size == 2 and s[1] == np.float32(2.0 / qmax)
    assert oracle.unpack_codes(c, 10, bits)[9] == -qmax
    assert np.array_equal(oracle.unpack_codes(c, 10, bits)[8:],
                          brute_force_codes(x[8:], s[1], qmax))


def test_subnormal_scale_is_honoured():
    # absmax tiny enough that s = absmax/127 is an fp32 subnormal
    x = np.array([2.0 ** -130, -2.0 ** -131, 2.0 ** -133], dtype=np.float32)
    c, s = oracle.block_quant(x, 3, 8)
    assert 0 < s[0] < np.finfo(np.float32).tiny
    assert np.array_equal(oracle.unpack_codes(c, 3, 8), brute_force_codes(x, s[0], 127))


def test_bf16_round_to_nearest_even_matches_torch():
    vals = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * 10.0 ** RNG.uniform(-30, 30, 20000),
        # exact ties between two bf16 neighbours, both parities
        ((np.arange(1000, dtype=np.uint32) << 16) | 0x8000).view(np.float32) + 0,
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40], np.float32),
    ]).astype(np.float32)
    vals = vals[np.isfinite(vals)]
    ours = oracle.f32_to_bf16(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---- a1/a2: qwZ shards ------------------------------------------------------------

def test_qwz_blocks_restart_at_every_shard():
    shard, block = 300, 256
    x = np.ones(2 * shard, np.float32)
    x[shard - 1] = 127.0                 # large value at the end of shard 0
    x[shard:] = 2.0                      # shard 1 is small
    xb = oracle.f32_to_bf16(x)
    codes, scales = oracle.qwz_quant(xb, 2, shard, block, 8)
    assert scales.size == 4
    assert scales[1] == 1.0                             # shard 0 tail block sees 127
    assert scales[2] == np.float32(2.0 / 127.0)         # shard 1 first block does not
    q = oracle.unpack_codes(codes, 2 * shard, 8)
    assert np.all(q[shard:] == 127)
    y = oracle.qwz_dequant(codes, scales, 2, shard, block, 8)
    assert y[shard - 1] == oracle.f32_to_bf16([127.0])[0]


def test_qwz_dequant_bound_and_bf16_rounding():
    nranks, shard, block = 3, 1000, 128
    w = (RNG.standard_normal(nranks * shard) * 0.02).astype(np.float32)
    wb = oracle.f32_to_bf16(w)
    xf = oracle.bf16_bits_to_f32(wb).astype(np.float64)
    for bits in (8, 4):
        qmax = (1 << (bits - 1)) - 1
        codes, scales = oracle.qwz_quant(wb, nranks, shard, block, bits)
        y = oracle.bf16_bits_to_f32(oracle.qwz_dequant(codes, scales, nranks, shard, block, bits))
        nb = -(-shard // block)
        s = np.concatenate([np.repeat(scales[r * nb:(r + 1) * nb].astype(np.float64), block)[:shard]
                            for r in range(nranks)])
        # s/2 from the code plus half a bf16 ulp (2^-8 relative) from the output rounding
        bound = s / 2 + 2 * 2.0 ** -24 * (qmax + 1) * s + np.abs(y) * 2.0 ** -8
        assert np.all(np.abs(y.astype(np.float64) - xf) <= bound)


# ---- O4: slice reordering ------------------------------------------------------------

def test_slice_perm_worked_example_and_identities():
    # N=2 nodes, G=3: position p = l*N + n holds slice j = n*G + l
    assert list(oracle.qgz_slice_perm(2, 3)) == [0, 3, 1, 4, 2, 5]
    for k in range(1, 9):
        assert list(oracle.qgz_slice_perm(1, k)) == list(range(k))
        assert list(oracle.qgz_slice_perm(k, 1)) == list(range(k))
    for N in range(1, 6):
        for G in range(1, 6):
            assert sorted(oracle.qgz_slice_perm(N, G)) == list(range(N * G))


def direct_reduce_scatter(grads_f64, Nd, bucket):
    """Textbook reduce-scatter with averaging: rank r gets the mean over ranks of
    slice r ("ZeRO Stage 2: Gradient Partitioning", Reduce-Scatter step 2)."""
    L = bucket // Nd
    g = grads_f64.reshape(Nd, Nd, L)
    return g.sum(axis=0)  # [slice r][i]; divided by Nd by the caller


@pytest.mark.parametrize("N", [1, 2, 3, 4])
@pytest.mark.parametrize("G", [1, 2, 3, 4])
def test_two_hop_placement_equals_reduce_scatter(N, G):
    """Identity codec + small-integer inputs: every sum is exact, so the two-hop
    chain must reproduce the direct reduce-scatter exactly."""
    Nd, L = N * G, 16
    bucket = Nd * L
    vals = RNG.integers(-50, 51, size=Nd * bucket).astype(np.float32)
    gb = oracle.f32_to_bf16(vals)
    got = oracle.qgz_reduce_scatter(gb, N, G, bucket, L, 32)
    sums = direct_reduce_scatter(vals.astype(np.float64), Nd, bucket)
    inv = np.float32(1.0) / np.float32(Nd)
    want = (sums.astype(np.float32) * inv).reshape(-1)
    assert np.array_equal(got, want)
    if Nd & (Nd - 1) == 0:   # power of two: the average itself is exact
        assert np.array_equal(got.astype(np.float64), (sums / Nd).reshape(-1))


@pytest.mark.parametrize("N,G", [(2, 2), (2, 3), (3, 2), (3, 4)])
def test_hop1_message_is_the_node_local_partial_sum(N, G):
    """Identity codec: after the intra-node all-to-all and reduction, rank
    (n, l) holds, in slot k, the sum over the G ranks of node n (ranks n*G..n*G+G-1)
    of slice k*G + l -- the part of rank (k, l)'s slice that node n contributes."""
    Nd, L = N * G, 8
    bucket = Nd * L
    vals = RNG.integers(-50, 51, size=Nd * bucket).astype(np.float32)
    codes, scales = oracle.qgz_reorder_quant(oracle.f32_to_bf16(vals), N, G, bucket, L, 32)
    c1, _ = oracle.qgz_hop1(codes, scales, N, G, bucket, L, 32)
    x = vals.reshape(N, G, Nd, L)            # [node][local][slice][i]
    c1 = c1.reshape(N, G, N, L)              # [node][local][slot][i]
    for n in range(N):
        for l in range(G):
            for k in range(N):
                assert np.array_equal(c1[n, l, k], x[n, :, k * G + l].sum(axis=0))


@pytest.mark.parametrize("N,G", [(2, 2), (2, 3), (3, 2), (4, 4)])
def test_without_reorder_slices_are_misplaced(N, G):
    Nd, L = N * G, 8
    bucket = Nd * L
    vals = RNG.integers(-50, 51, size=Nd * bucket).astype(np.float32)
    gb = oracle.f32_to_bf16(vals)
    codes, scales = oracle.qgz_reorder_quant(gb, N, G, bucket, L, 32,
                                             perm=np.arange(Nd, dtype=np.int32))
    c1, s1 = oracle.qgz_hop1(codes, scales, N, G, bucket, L, 32)
    got = oracle.qgz_hop2(c1, s1, N, G, bucket, L, 32)
    want = (direct_reduce_scatter(vals.astype(np.float64), Nd, bucket).astype(np.float32)
            * (np.float32(1) / np.float32(Nd))).reshape(-1)
    wrong = [r for r in range(Nd) if not np.array_equal(got[r * L:(r + 1) * L], want[r * L:(r + 1) * L])]
    assert wrong, "without the reorder some rank must receive another rank's slice"


def test_hop_sum_is_in_rank_order():
    """fp32: (0 + 2^24) + 1 = 2^24 (ties to even), then - 2^24 = 0; any other
    order of the three terms gives 1 or 2^24 + ... so only rank order gives 0."""
    N, G, L = 1, 3, 4
    Nd, bucket = 3, 12
    vals = np.zeros((Nd, bucket), np.float32)
    vals[0, :] = 2.0 ** 24
    vals[1, :] = 1.0
    vals[2, :] = -(2.0 ** 24)
    got = oracle.qgz_reduce_scatter(oracle.f32_to_bf16(vals.reshape(-1)), N, G, bucket, L, 32)
    assert np.all(got == 0.0)
    vals[[0, 1]] = vals[[1, 0]]          # 1 first: (1 + 2^24) = 2^24 ... also 0
    got = oracle.qgz_reduce_scatter(oracle.f32_to_bf16(vals.reshape(-1)), N, G, bucket, L, 32)
    assert np.all(got == 0.0)
    vals[[1, 2]] = vals[[2, 1]]          # 2^24 - 2^24 + 1 = 1
    got = oracle.qgz_reduce_scatter(oracle.f32_to_bf16(vals.reshape(-1)), N, G, bucket, L, 32)
    assert np.all(got == np.float32(1.0) * (np.float32(1) / np.float32(3)))


# ---- O3-O5 with the real codecs --------------------------------------------------------

@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,G", [(1, 4), (2, 2), (2, 4), (4, 2)])
def test_identical_exact_gradients_average_to_themselves(bits, N, G):
    """Every rank holds the same bucket, each block exactly q*s0 with s0 a power
    of two and one element at +-qmax: hop-1 requant and both averages are exact,
    so the reduce-scatter returns each rank's own slice unchanged."""
    qmax = (1 << (bits - 1)) - 1
    Nd, block = N * G, 64
    L = 2 * block
    bucket = Nd * L
    s0 = 2.0 ** -12
    q = RNG.integers(-qmax, qmax + 1, size=bucket)
    q[::block] = qmax * RNG.choice([-1, 1], size=bucket // block)
    x = (q * s0).astype(np.float32)
    gb = oracle.f32_to_bf16(np.tile(x, Nd))
    got = oracle.qgz_reduce_scatter(gb, N, G, bucket, block, bits)
    assert np.array_equal(got, x)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,G", [(1, 8), (2, 2), (2, 4), (3, 2), (4, 4)])
def test_reduce_scatter_error_bound(bits, N, G):
    Nd, block = N * G, 64
    L = 3 * block
    bucket = Nd * L
    x = (RNG.standard_normal(Nd * bucket) * 1e-3).astype(np.float32)
    gb = oracle.f32_to_bf16(x)
    xf = oracle.bf16_bits_to_f32(gb).astype(np.float64).reshape(Nd, Nd, L)   # [rank][slice][i]
    exact = xf.sum(axis=0) / Nd                                              # [slice r][i]
    codes, scales = oracle.qgz_reorder_quant(gb, N, G, bucket, block, bits)
    sc = scales.reshape(Nd, bucket // block).astype(np.float64)
    perm = oracle.qgz_slice_perm(N, G)
    pos = np.argsort(perm)                       # slice j -> position
    # per-element bound: half a scale for every quantization the value went through
    e1 = np.zeros((Nd, L))
    for r in range(Nd):
        for j in range(Nd):
            p = pos[j]
            e1[j] += np.repeat(sc[r, p * L // block:(p + 1) * L // block], block) / 2
    if N == 1:
        got = oracle.qgz_hop1(codes, scales, N, G, bucket, block, bits)
        e2 = np.zeros((Nd, L))
    else:
        c1, s1 = oracle.qgz_hop1(codes, scales, N, G, bucket, block, bits)
        got = oracle.qgz_hop2(c1, s1, N, G, bucket, block, bits)
        s1 = s1.reshape(Nd, N * L // block).astype(np.float64)
        e2 = np.zeros((Nd, L))
        for n in range(N):
            for l in range(G):
                d = n * G + l
                for n2 in range(N):
                    src = n2 * G + l
                    e2[d] += np.repeat(s1[src, n * L // block:(n + 1) * L // block], block) / 2
    qmax = (1 << (bits - 1)) - 1
    slack = (2 * Nd + 4) * 2.0 ** -23 * (np.abs(xf).sum(axis=0) + e1 + e2 + 1e-30) \
        + 2 * 2.0 ** -24 * (qmax + 1) * (e1 + e2)
    bound = (e1 + e2) / Nd + slack
    err = np.abs(got.reshape(Nd, L).astype(np.float64) - exact)
    assert np.all(err <= bound)


# ---- O6: Adam ---------------------------------------------------------------------------

def test_adam_first_step_closed_form():
    n = 5000
    g = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    g[:10] = 0.0
    p0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    lr, b1, b2, eps = 1e-4, 0.9, 0.999, 1e-8
    z = np.zeros(n, np.float32)
    p, m, v, pb = oracle.adam_step(g, p0, z, z, lr, b1, b2, eps, 1)
    b1f, b2f = np.float64(np.float32(b1)), np.float64(np.float32(b2))
    gd = g.astype(np.float64)
    # m' = (1 - b1) g, v' = (1 - b2) g^2 (each within a couple of roundings)
    assert np.allclose(m, (1 - b1f) * gd, rtol=3e-7, atol=0)
    assert np.allclose(v, (1 - b2f) * gd * gd, rtol=5e-7, atol=0)
    # bias corrections cancel: p' = p - lr g / (|g| + eps)
    want = p0.astype(np.float64) - lr * gd / (np.abs(gd) + eps)
    # the update term lr*g/(|g|+eps) carries a few fp32 roundings (relative
    # 2^-24 each) and the result one more
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(p - want) <= 2 * ulp + 8 * 2.0 ** -24 * lr)
    assert np.all(p[:10] == p0[:10])               # zero gradient: no move
    # the 16-bit write-back is the rounded master
    assert np.array_equal(pb, oracle.f32_to_bf16(p))


def test_adam_later_steps_against_double():
    """Each step against a float64 recomputation of the textbook update from
    the same fp32 state; error bounded by a few roundings of each term."""
    n = 3000
    u = 2.0 ** -24
    lr, b1, b2, eps = 3e-4, 0.9, 0.95, 1e-6
    p = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    m = (RNG.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(RNG.standard_normal(n) * 1e-6).astype(np.float32)
    b1f, b2f = float(np.float32(b1)), float(np.float32(b2))
    for t in (2, 3, 10, 1000):
        g = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
        pd, md, vd, gd = (a.astype(np.float64) for a in (p, m, v, g))
        p, m, v, _ = oracle.adam_step(g, p, m, v, lr, b1, b2, eps, t)
        mw = b1f * md + (1 - b1f) * gd
        vw = b2f * vd + (1 - b2f) * gd * gd
        mh, vh = mw / (1 - b1f ** t), vw / (1 - b2f ** t)
        upd = lr * mh / (np.sqrt(vh) + eps)
        pw = pd - upd
        assert np.all(np.abs(m - mw) <= 3 * u * (b1f * np.abs(md) + (1 - b1f) * np.abs(gd)) + 1e-45)
        assert np.all(np.abs(v - vw) <= 4 * u * (b2f * vd + (1 - b2f) * gd * gd) + 1e-45)
        assert np.all(np.abs(p - pw) <= u * np.abs(pw) + 12 * u * np.abs(upd) + 1e-45)
        # and the whole trajectory stays a 1e-5-relative match of the textbook values
        assert np.allclose(m, mw, rtol=1e-5, atol=1e-5 * np.abs(gd).max())


def test_adam_bias_constants():
    bc1, bc2, o1, o2 = oracle.adam_consts(0.9, 0.999, 1)
    assert bc1 == np.float32(1 - np.float64(np.float32(0.9)))
    assert o1 == bc1 and o2 == bc2
    bc1, bc2, _, _ = oracle.adam_consts(0.9, 0.999, 7)
    assert bc1 == np.float32(1 - np.float64(np.float32(0.9)) ** 7)
    assert bc2 == np.float32(1 - np.float64(np.float32(0.999)) ** 7)


# ---- O7: accounting ----------------------------------------------------------------------

def test_message_sizes_match_oracle_arrays():
    n, block = 10_000, 256
    x = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    for bits in (8, 4):
        c, s = oracle.block_quant(x, block, bits)
        assert c.nbytes + s.nbytes == accounting.quantized_bytes(n, block, bits)


def test_volume_fractions_match_pages():
    gv = golden("zeropp_volume.txt")
    z3 = accounting.zero3_volume()
    assert z3["fwd"] == Fraction(gv["zero3_fwd_allgather_M"])
    assert z3["bwd"] == Fraction(gv["zero3_bwd_allgather_M"])
    assert z3["grad"] == Fraction(gv["zero3_reduce_scatter_M"])
    assert z3["total"] == Fraction(gv["zero3_total_M"])
    phi = 7 * 10 ** 9
    for B in (64, 256, 512, 2048, 4096):
        v = accounting.zeropp_volume(phi - phi % B, B, 8, B, 4)
        # codes exactly the printed fractions, plus 4 B of scale per B elements
        assert v["fwd"] == Fraction(gv["qwz_fwd_M"]) + Fraction(2, B)
        assert v["grad"] == Fraction(gv["qgz_grad_M"]) + Fraction(2, B)
        assert v["bwd"] == Fraction(gv["hpz_bwd_cross_node_M"])
        assert v["total"] == Fraction(gv["zeropp_total_M"]) + Fraction(4, B)
        assert z3["total"] / v["total"] < 4 and abs(z3["total"] / v["total"] - 4) < 100 / B
    assert Fraction(gv["stage3_per_gpu_phi"]) / Fraction(gv["dp_per_gpu_phi"]) == \
        Fraction(gv["stage3_vs_dp_ratio"])


def test_memory_formulas_match_pages():
    gm = golden("zero_memory.txt")
    GB = 10 ** 9
    assert accounting.rank_memory(0, 175 * GB, 64) == int(gm["dp_175B_GB"]) * GB
    assert accounting.rank_memory(0, 7 * GB, 64) == int(gm["dp_7B_GB"]) * GB
    assert accounting.rank_memory(0, 1, 1) == int(gm["bytes_per_param_dp"])
    for nd in (1, 2, 8, 64, 1000):
        phi = 7 * GB
        assert accounting.rank_memory(1, phi, nd) == 4 * phi + Fraction(12 * phi, nd)
        assert accounting.rank_memory(2, phi, nd) == 2 * phi + Fraction(14 * phi, nd)
        assert accounting.rank_memory(3, phi, nd) == Fraction(16 * phi, nd)
    s2 = accounting.rank_memory(2, 7 * GB, 64)
    assert s2 == Fraction(gm["stage2_7B_nd64_formula_GB"]) * GB
    # the page's "14 GB of parameters" is the full 16-bit replica
    assert accounting.rank_buffers(2, 7 * GB, 64)[0].nbytes == int(gm["stage2_7B_nd64_params_GB"]) * GB
    # the page's printed total (14.9 GB) disagrees with its own formula
    assert s2 != Fraction(gm["stage2_7B_nd64_page_total_GB"]) * GB
    assert accounting.rank_memory(3, 7 * GB, 64) == Fraction(175, 100) * GB


def test_two_hop_avoids_cross_node_blow_up():
    for N, G in ((2, 8), (8, 8), (16, 8), (4, 2)):
        c = accounting.cross_node_bytes(N, G, N * G * 4096, 256, 4)
        assert c["flat"] == G * c["two_hop"]
    c = accounting.cross_node_bytes(1, 8, 8 * 4096, 256, 4)
    assert c["two_hop"] == 0 and c["flat"] == 0


# ---- O8: block vs global quantization ------------------------------------------------------

@pytest.mark.parametrize("bits", [8, 4])
def test_block_quantization_beats_global(bits):
    import synth
    from synth import workloads as W
    for recipe in (W.WEIGHT_RECIPE, W.GRAD_NORMAL, W.GRAD_T3_OUTLIERS):
        x = synth.fill(recipe, 0, synth.WEIGHTS, 0, 1 << 16).float().numpy()
        e = accounting.quant_errors(x, 256, bits)
        assert e["block"]["rmse"] <= e["global"]["rmse"]
        assert e["rmse_ratio"] > 1.0


# ---- next row: Adam -> qwZ of the new parameters ----------------------------------------------

def test_adam_then_qwz_message_bounds_and_shard_restart():
    nd, L, block = 4, 3 * 128, 128
    n = nd * L
    g = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    p0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    p0[L - 1] = 5.0                      # a large weight at the end of rank 0's shard
    z = np.zeros(n, np.float32)
    master, m, v, param, codes, scales = oracle.adam_then_qwz(
        g, p0, z, z, 1e-4, 0.9, 0.999, 1e-8, 1, nd, L, block)
    pf = oracle.bf16_bits_to_f32(param).astype(np.float64)
    nb = L // block
    s = np.repeat(scales.astype(np.float64), block)
    y = oracle.block_dequant(codes, scales, n, block, 8).astype(np.float64)
    # the message dequantizes to within s/2 (plus rounding) of the new 16-bit parameters
    assert np.all(np.abs(y - pf) <= s / 2 + 2 * 2.0 ** -24 * 128 * s)
    # rank 0's last block sees the large weight, rank 1's first block does not
    assert scales[nb - 1] >= np.float32(4.9 / 127)
    assert scales[nb] < np.float32(0.2 / 127)
    # the 16-bit parameters are the rounded masters of the Adam step
    assert np.array_equal(param, oracle.f32_to_bf16(master))


# ---- next row: gradient accumulation before the one-shot quantization ----------------------------

def test_accumulation_of_exact_microbatches_equals_quantizing_the_sum():
    """Small-integer micro-batches: the fp32 accumulation is exact, so
    accumulate-then-quantize equals quantizing the exact (float64) sum, and the
    identity codec returns the sum itself."""
    N, G, block = 2, 2, 64
    Nd, L = N * G, 2 * 64
    bucket = Nd * L
    mbs = [RNG.integers(-40, 41, size=Nd * bucket).astype(np.float32) for _ in range(5)]
    acc = oracle.grad_accumulate([oracle.f32_to_bf16(m) for m in mbs])
    exact = np.sum(np.stack(mbs).astype(np.float64), axis=0)
    assert np.array_equal(acc.astype(np.float64), exact)
    for bits in (8, 4):
        c, s = oracle.qgz_reorder_quant_f32(acc, N, G, bucket, block, bits)
        c2, s2 = oracle.qgz_reorder_quant_f32(exact.astype(np.float32), N, G, bucket, block, bits)
        assert np.array_equal(c, c2) and np.array_equal(s, s2)
    ident, _ = oracle.qgz_reorder_quant_f32(acc, N, G, bucket, L, 32)
    perm = oracle.qgz_slice_perm(N, G)
    x = exact.reshape(Nd, Nd, L)
    assert np.array_equal(ident.reshape(Nd, Nd, L), x[:, perm, :].astype(np.float32))


def test_accumulation_is_in_arrival_order():
    """(2^24 + 1) - 2^24 = 0 in fp32 when the 1 comes second, 1 when it comes last."""
    big, one = oracle.f32_to_bf16([2.0 ** 24]), oracle.f32_to_bf16([1.0])
    nbig = oracle.f32_to_bf16([-(2.0 ** 24)])
    assert oracle.grad_accumulate([big, one, nbig])[0] == 0.0
    assert oracle.grad_accumulate([big, nbig, one])[0] == 1.0


def test_bf16_bucket_quantizes_like_its_fp32_widening():
    """The fp32-input quantizer on widened bf16 values equals the bf16 one."""
    N, G, block = 2, 4, 128
    Nd, L = N * G, 3 * 128
    bucket = Nd * L
    gb = oracle.f32_to_bf16((RNG.standard_normal(Nd * bucket) * 1e-3).astype(np.float32))
    for bits in (8, 4):
        a = oracle.qgz_reorder_quant(gb, N, G, bucket, block, bits)
        b = oracle.qgz_reorder_quant_f32(oracle.bf16_bits_to_f32(gb), N, G, bucket, block, bits)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- next row: hpZ secondary partition and node-local backward gather ------------------------------

def test_hpz_gather_hand_worked():
    """G = 2 ranks, N = 2 shards each, shard = 4, block = 2, int8: the
    gathered weights are q * s for hand-picked codes and power-of-two scales."""
    codes = [np.array([1, -2, 3, 4, -5, 6, 7, -8], np.int8).view(np.uint8),
             np.array([10, 0, -1, 2, 127, -127, 64, 32], np.int8).view(np.uint8)]
    scales = [np.array([0.5, 0.25, 1.0, 2.0], np.float32),
              np.array([0.125, 4.0, 2.0 ** -7, 1.0], np.float32)]
    y = oracle.hpz_gather(list(zip(codes, scales)), 2, 4, 2, 8)
    want = [0.5, -1.0, 0.75, 1.0, -5.0, 6.0, 14.0, -16.0,
            1.25, 0.0, -4.0, 8.0, 127 / 128, -127 / 128, 64.0, 32.0]
    assert np.array_equal(oracle.bf16_bits_to_f32(y), np.array(want, np.float32))


@pytest.mark.parametrize("bits", [8, 4, 16])
@pytest.mark.parametrize("N,G", [(1, 8), (2, 4), (4, 2), (3, 3)])
def test_hpz_gather_of_kept_forward_messages_is_the_forward_gather(bits, N, G):
    """The secondary partitions are the forward all-gather's messages of the
    node's slices; gathering them in local rank order rebuilds exactly the
    weights the forward all-gather delivered, and a swap of two ranks'
    secondaries shows in the result."""
    Nd, shard, block = N * G, 3 * 256 + 64, 128
    w = oracle.f32_to_bf16((RNG.standard_normal(Nd * shard) * 0.02).astype(np.float32))
    if bits == 16:
        fwd = w
        secs = [w[l * N * shard:(l + 1) * N * shard].copy() for l in range(G)]
    else:
        c, s = oracle.qwz_quant(w, Nd, shard, block, bits)
        fwd = oracle.qwz_dequant(c, s, Nd, shard, block, bits)
        cb, nb = oracle.codes_bytes(shard, bits), oracle.num_blocks(shard, block)
        secs = [(c[l * N * cb:(l + 1) * N * cb].copy(), s[l * N * nb:(l + 1) * N * nb].copy())
                for l in range(G)]
    y = oracle.hpz_gather(secs, N, shard, block, bits)
    assert np.array_equal(y, fwd)
    if G > 1:
        secs[0], secs[1] = secs[1], secs[0]
        assert not np.array_equal(oracle.hpz_gather(secs, N, shard, block, bits), fwd)


def test_hpz_secondary_memory_is_a_node_replica():
    """Each rank keeps Phi/G of the weights (codes + scales); the G ranks of a
    node together hold one full replica, the memory the pages trade for the
    zero cross-node backward volume."""
    for N, G in ((1, 8), (2, 8), (8, 8), (16, 8)):
        Nd = N * G
        for block, bits in ((256, 8), (2048, 8), (512, 4)):
            shard = 64 * block
            phi = Nd * shard
            per_rank = oracle.hpz_secondary_bytes(N, shard, block, bits)
            assert per_rank == Fraction(phi, G) * Fraction(bits, 8) + 4 * Fraction(phi, G * block)
            assert G * per_rank == accounting.quantized_bytes(phi, block, bits)
            assert oracle.hpz_secondary_bytes(N, shard, block, 16) == 2 * phi // G
    gv = golden("zeropp_volume.txt")
    assert Fraction(gv["hpz_bwd_cross_node_M"]) == 0


# ---- next row: ring reduce-scatter with a requantization per hop (precision comparator) ----------

@pytest.mark.parametrize("nd", [1, 2, 3, 4, 8])
def test_ring_with_identity_codec_is_the_average(nd):
    """Small integers sum exactly in fp32, so with the identity codec rank r
    ends with sum_k x_k[chunk r] * fl(1/N_d), whatever the ring order."""
    L, block = 3 * 64, 64
    bucket = nd * L
    xi = RNG.integers(-50, 51, size=(nd, nd, L))
    x = oracle.f32_to_bf16(xi.astype(np.float32).reshape(-1))
    g = oracle.ring_reduce_scatter(x, nd, bucket, block, 32)
    want = xi.sum(axis=0).astype(np.float32) * np.float32(1.0 / nd)
    assert np.array_equal(g.reshape(nd, L), want)


def test_ring_two_ranks_composed_from_block_codec():
    """N_d = 2: chunk 0 goes 1 -> 0, so g_0 = (D(Q(x_1[0])) + x_0[0]) * 0.5 and
    g_1 = (D(Q(x_0[1])) + x_1[1]) * 0.5."""
    L, block = 4 * 64, 64
    x = oracle.f32_to_bf16((RNG.standard_normal(2 * 2 * L) * 1e-3).astype(np.float32))
    xf = oracle.bf16_bits_to_f32(x).reshape(2, 2, L)
    for bits in (8, 4):
        g = oracle.ring_reduce_scatter(x, 2, 2 * L, block, bits).reshape(2, L)
        for r in (0, 1):
            c, s = oracle.block_quant(xf[1 - r, r], block, bits)
            d = oracle.block_dequant(c, s, L, block, bits)
            want = (d + xf[r, r]) * np.float32(0.5)
            assert np.array_equal(g[r], want.astype(np.float32))


@pytest.mark.parametrize("nd", [3, 8])
def test_ring_error_within_the_sum_of_half_scales(nd):
    """Chunk c passes N_d - 1 quantizations on its way round the ring; each
    moves an element by at most half its block's scale, so the result is
    within (sum of those half scales) / N_d of the exact average (plus fp32
    rounding of the adds)."""
    L, block, bits = 2 * 128, 128, 4
    bucket = nd * L
    x = oracle.f32_to_bf16((RNG.standard_normal(nd * bucket) * 1e-3).astype(np.float32))
    xf = oracle.bf16_bits_to_f32(x).reshape(nd, nd, L).astype(np.float64)
    nb = L // block
    half = np.zeros((nd, nb))          # per chunk, per block: sum of s/2 along the ring
    ci = si = None
    for step in range(nd):
        out = oracle.ring_rs_step(step, nd, bucket, block, bits, x, ci, si)
        if step == nd - 1:
            g = out.reshape(nd, L)
            break
        ci, si = out
        for r in range(nd):
            c = (r - 1 - step) % nd
            half[c] += si.reshape(nd, nb)[r] / 2
    exact = xf.sum(axis=0) / nd
    bound = np.repeat(half, block, axis=1) / nd + 1e-6 * np.abs(xf).sum(axis=0).max()
    assert np.all(np.abs(g - exact) <= bound)
    assert np.any(np.abs(g - exact) > 0.1 * bound)   # the bound is not vacuous


def test_ring_error_grows_with_nd_and_exceeds_qgz():
    """The pages' point: N sequential requantizations lose precision that the
    one-shot quantization of qgZ does not.  On seeded N(0, 1e-3) gradients the
    ring's relative RMS error grows with N_d while qgZ's stays flat."""
    rng = np.random.default_rng(3)
    block, bits = 256, 4
    ring, qgz = [], []
    for nd in (2, 4, 8, 16, 32):
        L = 4 * block
        bucket = nd * L
        x = oracle.f32_to_bf16((rng.standard_normal(nd * bucket) * 1e-3).astype(np.float32))
        xf = oracle.bf16_bits_to_f32(x).reshape(nd, nd, L).astype(np.float64)
        exact = (xf.sum(axis=0) / nd).reshape(-1)
        rms = np.sqrt(np.mean(exact ** 2))
        N, G = (1, nd) if nd <= 8 else (nd // 8, 8)
        gr = oracle.ring_reduce_scatter(x, nd, bucket, block, bits)
        gq = oracle.qgz_reduce_scatter(x, N, G, bucket, block, bits)
        ring.append(np.sqrt(np.mean((gr - exact) ** 2)) / rms)
        qgz.append(np.sqrt(np.mean((gq - exact) ** 2)) / rms)
    assert all(b > a for a, b in zip(ring, ring[1:]))
    assert max(qgz) < 1.6 * min(qgz)
    assert ring[2] > 1.5 * qgz[2] and ring[4] > 2.5 * qgz[4]


def test_ring_sums_in_ring_order():
    """N_d = 4, identity codec: chunk 0 is summed by ranks 1, 2, 3, then 0.
    With x_1 = 2^24, x_2 = x_3 = 1, x_0 = -2^24 that order loses both ones
    ((2^24 + 1) rounds to 2^24) and gives 0; the reverse ring direction
    (3, 2, 1, 0) would give 2 / 4."""
    nd, L, block = 4, 64, 64
    xf = np.zeros((nd, nd, L), np.float32)
    xf[1, 0], xf[2, 0], xf[3, 0], xf[0, 0] = 2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)
    x = oracle.f32_to_bf16(xf.reshape(-1))
    g = oracle.ring_reduce_scatter(x, nd, nd * L, block, 32).reshape(nd, L)
    assert np.all(g[0] == 0.0)
    assert np.all(g[1:] == 0.0)
