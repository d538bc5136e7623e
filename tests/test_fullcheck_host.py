"""CPU tests of the complete full-size checkers (tests/fullcheck.py): on a
small pass whose outputs the oracle itself wrote into CPU tensors laid out
like CodecPath's buffers, the piecewise checks (qwZ shards split at block
boundaries, qgZ and ring buckets split into groups of block positions) pass,
and a single planted wrong byte or value anywhere is found."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import fullcheck as F
import oracle
import synth
from synth import workloads as W


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def fake_qgz_path(N, G, L, B, bits, seed, microbatches=1, adam=True, fuse_qwz=False):
    """A CodecPath-shaped namespace holding the oracle's outputs of one pass."""
    nd, bucket = N * G, N * G * L
    recipe = W.GRAD_T3_OUTLIERS
    mbs = [np.concatenate([synth.fill_u16(recipe, seed, synth.grad_stream(r, k), 0, bucket)
                           for r in range(nd)]) for k in range(microbatches)]
    if microbatches == 1:
        c1, s1 = oracle.qgz_reorder_quant(mbs[0], N, G, bucket, B, bits)
    else:
        c1, s1 = oracle.qgz_reorder_quant_f32(oracle.grad_accumulate(mbs), N, G, bucket, B, bits)
    p = SimpleNamespace(qgz=SimpleNamespace(nodes=N, gpus_per_node=G, nd=nd, L=L, block=B,
                                            bits=bits, bucket=bucket),
                        microbatches=microbatches, fuse_qwz=fuse_qwz, adam=None, param=None,
                        msg1=_t(c1), msg1_scales=_t(s1), standalone_adam=0, qwz=None)
    if microbatches > 1:
        p.acc = _t(oracle.grad_accumulate(mbs[:-1]))
    if N > 1:
        c2, s2 = oracle.qgz_hop1(c1, s1, N, G, bucket, B, bits)
        p.msg2, p.msg2_scales = _t(c2), _t(s2)
        g = oracle.qgz_hop2(c2, s2, N, G, bucket, B, bits)
    else:
        g = oracle.qgz_hop1(c1, s1, N, G, bucket, B, bits)
    p.grad_out = _t(g)
    wl = SimpleNamespace(seed=seed, qgz=SimpleNamespace(grad=recipe), adam=W.Adam())
    if adam:
        a = wl.adam
        p.adam = a
        p0 = F.widen(synth.fill_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, 0, bucket))
        z = np.zeros(bucket, np.float32)
        wp, wm, wv, wb = oracle.adam_step(g, p0, z, z, a.lr, a.beta1, a.beta2, a.eps, a.step)
        p.master, p.m, p.v, p.param = _t(wp), _t(wm), _t(wv), _t(wb)
        if fuse_qwz:
            wc, ws = oracle.qwz_quant(wb, nd, L, B, 8)
            p.w_codes, p.w_scales = [_t(wc)], [_t(ws)]
    return p, wl


@pytest.fixture(autouse=True)
def small_pieces(monkeypatch):
    monkeypatch.setattr(F, "GROUP_ELEMS", 1 << 12)
    monkeypatch.setattr(F, "QWZ_PIECE", 1 << 10)


@pytest.mark.parametrize("N,G,bits,mb,fuse", [(2, 2, 4, 1, False), (1, 4, 4, 1, True),
                                              (3, 2, 8, 2, False), (2, 3, 4, 3, False)])
def test_qgz_checker_passes_on_oracle_outputs(N, G, bits, mb, fuse):
    p, wl = fake_qgz_path(N, G, 6 * 64, 64, bits, seed=4, microbatches=mb, fuse_qwz=fuse)
    assert F.check_qgz_complete(p, wl) > 1      # several groups of block positions


@pytest.mark.parametrize("buf", ["msg1", "msg1_scales", "msg2", "msg2_scales", "grad_out",
                                 "master", "m", "v", "param", "acc"])
@pytest.mark.parametrize("where", [0.0, 0.37, 0.999])
def test_qgz_checker_finds_a_planted_error(buf, where):
    p, wl = fake_qgz_path(2, 2, 6 * 64, 64, 4, seed=5, microbatches=2)
    t = getattr(p, buf)
    flat = t.view(torch.uint8) if t.dtype == torch.uint8 else t.view(torch.int16) \
        if t.dtype == torch.bfloat16 else t.view(torch.int32)
    i = min(flat.numel() - 1, int(where * flat.numel()))
    # bytes: a changed code; bf16: 4 ulp; fp32 state: 256 ulp (above 1e-5 relative)
    flat[i] ^= 0x100 if buf in ("master", "m", "v") else 0x4 if buf == "param" else 0x3
    with pytest.raises(AssertionError):
        F.check_qgz_complete(p, wl)


def test_fused_qwz_codes_checked():
    p, wl = fake_qgz_path(1, 4, 4 * 64, 64, 4, seed=6, fuse_qwz=True)
    p.w_codes[0][-1] ^= 1
    with pytest.raises(AssertionError):
        F.check_qgz_complete(p, wl)


def fake_qwz_path(nranks, shards, block, bits, seed):
    q = SimpleNamespace(nranks=nranks, block=block, bits=bits, call_shards=lambda: shards)
    phi = nranks * sum(shards)
    w = synth.fill_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, 0, phi)
    sizes = sorted(set(shards))
    p = SimpleNamespace(qwz=q, _codes_of={s: i for i, s in enumerate(sizes)},
                        w_codes=[None] * len(sizes), w_scales=[None] * len(sizes),
                        w_full=_t(np.zeros(phi, np.uint16)))
    return p, SimpleNamespace(seed=seed), w


@pytest.mark.parametrize("bits", [8, 4])
def test_qwz_capture_checks_every_call(bits):
    shards = [3 * 1024, 3 * 1024, 1000]           # a streamed tensor with a short tail call
    p, wl, w = fake_qwz_path(2, shards, 256, bits, seed=7)
    cap = F.QwzCapture(p, wl)
    off = 0
    for k, s in enumerate(shards):
        n = 2 * s
        c, sc = oracle.qwz_quant(w[off:off + n], 2, s, 256, bits)
        y = oracle.qwz_dequant(c, sc, 2, s, 256, bits)
        if k == 1:               # plant one wrong code byte in the middle call
            c = c.copy()
            c[len(c) // 2] ^= 0x10
        p.w_codes[p._codes_of[s]], p.w_scales[p._codes_of[s]] = _t(c), _t(sc)
        p.w_full[off:off + n] = _t(y)
        cap("qwz_quant")
        cap("qwz_dequant")
        off += n
    with pytest.raises(AssertionError, match="call 1"):
        cap.finish()


def test_ring_checker():
    nd, L, B, bits = 4, 4 * 64, 64, 4
    q = W.QgZ(nodes=1, gpus_per_node=nd, bucket=nd * L, block=B, bits=bits)
    x = np.concatenate([synth.fill_u16(q.grad, 2, synth.grad_stream(r), 0, nd * L)
                        for r in range(nd)])
    g = oracle.ring_reduce_scatter(x, nd, nd * L, B, bits)
    F.check_ring_complete(_t(g), q, 2)
    g = g.copy()
    g[3 * L + 5] = np.nextafter(g[3 * L + 5], np.float32(1))
    with pytest.raises(AssertionError):
        F.check_ring_complete(_t(g), q, 2)


def test_adam_checker():
    n, seed, hp = 5000, 3, (1e-4, 0.9, 0.999, 1e-8, 7)
    g = F.widen(synth.fill_u16(W.GRAD_NORMAL, seed, 11, 0, n))
    p0 = F.widen(synth.fill_u16(W.WEIGHT_RECIPE, seed, synth.WEIGHTS, 0, n))
    m0 = F.widen(synth.fill_u16(W.MOMENT_M_RECIPE, seed, synth.MOMENT_M, 0, n))
    v0 = F.widen(synth.fill_u16(W.MOMENT_V_RECIPE, seed, synth.MOMENT_V, 0, n))
    wp, wm, wv, wb = oracle.adam_step(g, p0, m0, v0, *hp)
    dev = [_t(wp), _t(wm), _t(wv), _t(wb)]
    F.check_adam_complete(dev, n, seed, hp, W.GRAD_NORMAL, 11)
    dev[2] = _t(wv * np.float32(1.001))
    with pytest.raises(AssertionError):
        F.check_adam_complete(dev, n, seed, hp, W.GRAD_NORMAL, 11)
