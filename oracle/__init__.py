"""CPU oracle of the ZeRO++ data-parallel codec path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference leg are the only callers.  The product path
(the CUDA library and its binding) never imports this package, and this
package imports nothing from the product.

The arithmetic lives in ``zpp_oracle.c`` (plain single-threaded C, fp32 with
no FMA contraction, each function citing the passage it follows).  This module
only builds it with gcc, marshals numpy arrays and adds the byte accounting
(``accounting``).  Layout conventions are the ones the method states:

* qwZ: bf16 ``[nranks][shard]`` -> codes ``[nranks][ceil(shard*bits/8)]`` and
  fp32 scales ``[nranks][ceil(shard/block)]``.
* qgZ: bf16 ``[N_d][bucket]``; slice ``j = n*G + l`` of every bucket belongs
  to rank ``(n, l)``; the one-shot message stores slice ``j`` at position
  ``l*N + n``; hop-1 messages are ``[N_d][N*L]``; the final output is fp32
  ``[N_d][L]`` indexed by the global parameter index ``r*L + i``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zpp_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wextra"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (in-tree, next to its source)."""
    with _lock:
        stale = (not os.path.exists(_SO)
                 or os.path.getmtime(_SO) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _SO + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    try:
        lib = ctypes.CDLL(_SO)
    except OSError:  # e.g. a binary built for another machine
        build(force=True)
        lib = ctypes.CDLL(_SO)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    sig = {
        "orc_f32_to_bf16": (ctypes.c_uint16, [F]),
        "orc_codes_bytes": (I64, [I64, I32]),
        "orc_num_blocks": (I64, [I64, I64]),
        "orc_block_quant": (I32, [P, I64, I64, I32, P, P]),
        "orc_block_dequant": (I32, [P, P, I64, I64, I32, P]),
        "orc_qwz_quant": (I32, [P, I64, I64, I64, I32, P, P]),
        "orc_qwz_dequant": (I32, [P, P, I64, I64, I64, I32, P]),
        "orc_qgz_slice_perm": (I32, [I32, I32, P]),
        "orc_qgz_reorder_quant": (I32, [P, I32, I32, I64, I64, I32, P, P]),
        "orc_qgz_reorder_quant_perm": (I32, [P, I32, I32, I64, I64, I32, P, P, P]),
        "orc_qgz_hop1": (I32, [P, P, I32, I32, I64, I64, I32, P, P, P]),
        "orc_qgz_hop2": (I32, [P, P, I32, I32, I64, I64, I32, P]),
        "orc_adam_consts": (None, [F, F, I32, P, P, P, P]),
        "orc_adam_step": (I32, [P, I64, F, F, F, F, I32, P, P, P, P]),
        "orc_grad_accumulate": (I32, [P, P, I64, I32]),
        "orc_qgz_reorder_quant_f32": (I32, [P, I32, I32, I64, I64, I32, P, P]),
        "orc_hpz_gather": (I32, [I32, I32, I64, I64, I32, P, P, P]),
        "orc_hpz_secondary_bytes": (I64, [I32, I64, I64, I32]),
        "orc_ring_rs_step": (I32, [I32, I32, I64, I64, I32, P, P, P, P, P, P]),
        "orc_ring_reduce_scatter": (I32, [I32, I64, I64, I32, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# ---- sizes -------------------------------------------------------------------

def codes_bytes(n: int, bits: int) -> int:
    return int(_load().orc_codes_bytes(n, bits))


def num_blocks(n: int, block: int) -> int:
    return int(_load().orc_num_blocks(n, block))


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) of fp32 values, round to nearest even."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---- O1/O2 ------------------------------------------------------------------

def _code_dtype(bits):
    return np.float32 if bits == 32 else np.uint8


def block_quant(x: np.ndarray, block: int, bits: int):
    """O1 on a 1-D fp32 run: returns (codes, scales)."""
    x = _c(np.asarray(x, dtype=np.float32).reshape(-1), np.float32)
    n = x.size
    codes = np.zeros(n if bits == 32 else codes_bytes(n, bits), dtype=_code_dtype(bits))
    scales = np.zeros(max(num_blocks(n, block), 0), dtype=np.float32)
    _check(_load().orc_block_quant(_ptr(x), n, block, bits, _ptr(codes), _ptr(scales)),
           "block_quant")
    return codes, scales


def block_dequant(codes: np.ndarray, scales: np.ndarray, n: int, block: int, bits: int):
    """O2: fp32 values (float)q * s."""
    y = np.zeros(n, dtype=np.float32)
    codes = np.ascontiguousarray(codes)
    scales = _c(scales, np.float32)
    _check(_load().orc_block_dequant(_ptr(codes), _ptr(scales), n, block, bits, _ptr(y)),
           "block_dequant")
    return y


def unpack_codes(codes: np.ndarray, n: int, bits: int) -> np.ndarray:
    """Signed integer codes of a packed int8/int4 stream (for tests)."""
    codes = np.ascontiguousarray(codes).view(np.uint8)
    if bits == 8:
        return codes[:n].view(np.int8).astype(np.int32)
    lo = (codes & 0xF).astype(np.int32)
    hi = (codes >> 4).astype(np.int32)
    q = np.empty(2 * codes.size, dtype=np.int32)
    q[0::2], q[1::2] = lo, hi
    q = q[:n]
    return np.where(q >= 8, q - 16, q)


# ---- a1/a2: qwZ ---------------------------------------------------------------

def qwz_quant(x_bf16: np.ndarray, nranks: int, shard: int, block: int, bits: int):
    x = _c(x_bf16, np.uint16)
    assert x.size == nranks * shard
    codes = np.zeros(nranks * codes_bytes(shard, bits), dtype=np.uint8)
    scales = np.zeros(nranks * num_blocks(shard, block), dtype=np.float32)
    _check(_load().orc_qwz_quant(_ptr(x), nranks, shard, block, bits, _ptr(codes),
                                 _ptr(scales)), "qwz_quant")
    return codes, scales


def qwz_dequant(codes, scales, nranks: int, shard: int, block: int, bits: int):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    y = np.zeros(nranks * shard, dtype=np.uint16)
    _check(_load().orc_qwz_dequant(_ptr(codes), _ptr(scales), nranks, shard, block, bits,
                                   _ptr(y)), "qwz_dequant")
    return y


# ---- a3-a5: qgZ ---------------------------------------------------------------

def qgz_slice_perm(N: int, G: int) -> np.ndarray:
    perm = np.zeros(N * G, dtype=np.int32)
    _check(_load().orc_qgz_slice_perm(N, G, _ptr(perm)), "slice_perm")
    return perm


def qgz_reorder_quant(grads_bf16, N: int, G: int, bucket: int, block: int, bits: int,
                      perm: np.ndarray | None = None):
    g = _c(grads_bf16, np.uint16)
    Nd = N * G
    assert g.size == Nd * bucket
    if bits == 32:
        codes = np.zeros(Nd * bucket, dtype=np.float32)
    else:
        codes = np.zeros(Nd * codes_bytes(bucket, bits), dtype=np.uint8)
    scales = np.zeros(Nd * (bucket // block), dtype=np.float32)
    lib = _load()
    if perm is None:
        rc = lib.orc_qgz_reorder_quant(_ptr(g), N, G, bucket, block, bits, _ptr(codes),
                                       _ptr(scales))
    else:
        perm = _c(perm, np.int32)
        rc = lib.orc_qgz_reorder_quant_perm(_ptr(g), N, G, bucket, block, bits,
                                            _ptr(perm), _ptr(codes), _ptr(scales))
    _check(rc, "qgz_reorder_quant")
    return codes, scales


def qgz_hop1(codes_in, scales_in, N: int, G: int, bucket: int, block: int, bits: int):
    """Returns (codes_out, scales_out) when N > 1, else the final fp32 gradient."""
    Nd = N * G
    L = bucket // Nd
    codes_in = np.ascontiguousarray(codes_in)
    scales_in = _c(scales_in, np.float32)
    lib = _load()
    if N == 1:
        g = np.zeros(Nd * L, dtype=np.float32)
        _check(lib.orc_qgz_hop1(_ptr(codes_in), _ptr(scales_in), N, G, bucket, block, bits,
                                None, None, _ptr(g)), "qgz_hop1")
        return g
    NL = N * L
    if bits == 32:
        co = np.zeros(Nd * NL, dtype=np.float32)
    else:
        co = np.zeros(Nd * codes_bytes(NL, bits), dtype=np.uint8)
    so = np.zeros(Nd * (NL // block), dtype=np.float32)
    _check(lib.orc_qgz_hop1(_ptr(codes_in), _ptr(scales_in), N, G, bucket, block, bits,
                            _ptr(co), _ptr(so), None), "qgz_hop1")
    return co, so


def qgz_hop2(codes_in, scales_in, N: int, G: int, bucket: int, block: int, bits: int):
    Nd = N * G
    L = bucket // Nd
    codes_in = np.ascontiguousarray(codes_in)
    scales_in = _c(scales_in, np.float32)
    g = np.zeros(Nd * L, dtype=np.float32)
    _check(_load().orc_qgz_hop2(_ptr(codes_in), _ptr(scales_in), N, G, bucket, block, bits,
                                _ptr(g)), "qgz_hop2")
    return g


def qgz_reduce_scatter(grads_bf16, N: int, G: int, bucket: int, block: int, bits: int):
    """The whole qgZ chain: reorder+quant, hop 1, hop 2 (if N > 1)."""
    codes, scales = qgz_reorder_quant(grads_bf16, N, G, bucket, block, bits)
    if N == 1:
        return qgz_hop1(codes, scales, N, G, bucket, block, bits)
    c1, s1 = qgz_hop1(codes, scales, N, G, bucket, block, bits)
    return qgz_hop2(c1, s1, N, G, bucket, block, bits)


# ---- a6: Adam --------------------------------------------------------------------

def adam_consts(beta1: float, beta2: float, t: int):
    f = [ctypes.c_float() for _ in range(4)]
    _load().orc_adam_consts(beta1, beta2, t, *[ctypes.byref(x) for x in f])
    return tuple(x.value for x in f)  # bc1, bc2, 1-beta1, 1-beta2


def adam_step(g, master, m, v, lr, beta1, beta2, eps, t, want_param=True):
    """Returns updated (master, m, v, param_bf16_bits) as new arrays."""
    g = _c(g, np.float32)
    master = np.array(master, dtype=np.float32, copy=True)
    m = np.array(m, dtype=np.float32, copy=True)
    v = np.array(v, dtype=np.float32, copy=True)
    param = np.zeros(g.size, dtype=np.uint16) if want_param else None
    _check(_load().orc_adam_step(_ptr(g), g.size, lr, beta1, beta2, eps, t, _ptr(master),
                                 _ptr(m), _ptr(v), _ptr(param)), "adam_step")
    return master, m, v, param


# ---- next rows ---------------------------------------------------------------------

def adam_then_qwz(g, master, m, v, lr, beta1, beta2, eps, t, nd: int, L: int, block: int,
                  bits: int = 8):
    """Adam step on every rank's owned slice, then the qwZ message of the new
    16-bit parameters for the next forward all-gather ("ZeRO-1/2/3", Stage 1
    steps 6-7: write back the 16-bit parameters, all-gather them; "Quantized
    LLM Training at Scale with ZeRO++", 1 QWZ: that all-gather travels as
    block-quantized 8-bit codes).  Element d*L + i is parameter i of rank d's
    shard; blocks restart at every shard.
    Returns (master, m, v, param_bf16_bits, codes, scales)."""
    master, m, v, param = adam_step(g, master, m, v, lr, beta1, beta2, eps, t)
    codes, scales = qwz_quant(param, nd, L, block, bits)
    return master, m, v, param, codes, scales


def grad_accumulate(microbatches_bf16) -> np.ndarray:
    """fp32 sum of bf16 micro-batch gradients in arrival order (acc = g1;
    acc = acc + gk) -- the accumulator before the reduce-scatter ("ZeRO Stage 2:
    Gradient Partitioning", gradient accumulation)."""
    mbs = [_c(g, np.uint16) for g in microbatches_bf16]
    acc = np.zeros(mbs[0].size, dtype=np.float32)
    for k, g in enumerate(mbs):
        _check(_load().orc_grad_accumulate(_ptr(g), _ptr(acc), g.size, 1 if k == 0 else 0),
               "grad_accumulate")
    return acc


def qgz_reorder_quant_f32(grads_f32, N: int, G: int, bucket: int, block: int, bits: int):
    """The one-shot reorder + quantization of an fp32 bucket (accumulated gradients)."""
    g = _c(grads_f32, np.float32)
    Nd = N * G
    assert g.size == Nd * bucket
    if bits == 32:
        codes = np.zeros(Nd * bucket, dtype=np.float32)
    else:
        codes = np.zeros(Nd * codes_bytes(bucket, bits), dtype=np.uint8)
    scales = np.zeros(Nd * (bucket // block), dtype=np.float32)
    _check(_load().orc_qgz_reorder_quant_f32(_ptr(g), N, G, bucket, block, bits, _ptr(codes),
                                             _ptr(scales)), "qgz_reorder_quant_f32")
    return codes, scales


def hpz_gather(secondaries, N: int, shard: int, block: int, bits: int) -> np.ndarray:
    """Backward weight gather of one node under hpZ: `secondaries[l]` is local
    rank l's secondary partition, (codes, scales) of N consecutive primary
    shards, or a bf16 array of N*shard values when bits == 16.  Returns the
    full bf16 weights [G*N*shard]."""
    G = len(secondaries)
    keep = []
    cp = (ctypes.c_void_p * G)()
    sp = (ctypes.c_void_p * G)()
    for l, sec in enumerate(secondaries):
        if bits == 16:
            c = _c(sec, np.uint16)
            s = None
        else:
            c, s = sec
            c = np.ascontiguousarray(c)
            s = _c(s, np.float32)
        keep.append((c, s))
        cp[l] = c.ctypes.data
        sp[l] = None if s is None else s.ctypes.data
    y = np.zeros(G * N * shard, dtype=np.uint16)
    _check(_load().orc_hpz_gather(G, N, shard, block, bits, ctypes.cast(cp, ctypes.c_void_p),
                                  ctypes.cast(sp, ctypes.c_void_p), _ptr(y)), "hpz_gather")
    return y


def hpz_secondary_bytes(N: int, shard: int, block: int, bits: int) -> int:
    return int(_load().orc_hpz_secondary_bytes(N, shard, block, bits))


def ring_rs_step(step: int, nd: int, bucket: int, block: int, bits: int, grads_bf16,
                 codes_in=None, scales_in=None):
    """One step of the quantized ring reduce-scatter (the comparator of qgZ's
    one-shot quantization).  Returns (codes, scales), or the fp32 gradient
    [N_d][L] at the last step."""
    x = _c(grads_bf16, np.uint16)
    assert x.size == nd * bucket
    L = bucket // nd
    if step == nd - 1:
        g = np.zeros(nd * L, dtype=np.float32)
        _check(_load().orc_ring_rs_step(step, nd, bucket, block, bits, _ptr(x),
                                        _ptr(None if codes_in is None else np.ascontiguousarray(codes_in)),
                                        _ptr(None if scales_in is None else _c(scales_in, np.float32)),
                                        None, None, _ptr(g)), "ring_rs_step")
        return g
    if bits == 32:
        codes = np.zeros(nd * L, dtype=np.float32)
    else:
        codes = np.zeros(nd * codes_bytes(L, bits), dtype=np.uint8)
    scales = np.zeros(nd * num_blocks(L, block), dtype=np.float32)
    ci = None if codes_in is None else np.ascontiguousarray(codes_in)
    si = None if scales_in is None else _c(scales_in, np.float32)
    _check(_load().orc_ring_rs_step(step, nd, bucket, block, bits, _ptr(x), _ptr(ci), _ptr(si),
                                    _ptr(codes), _ptr(scales), None), "ring_rs_step")
    return codes, scales


def ring_reduce_scatter(grads_bf16, nd: int, bucket: int, block: int, bits: int) -> np.ndarray:
    """The whole quantized ring: rank r's averaged chunk r, [N_d][L] fp32."""
    x = _c(grads_bf16, np.uint16)
    assert x.size == nd * bucket
    g = np.zeros(bucket, dtype=np.float32)
    _check(_load().orc_ring_reduce_scatter(nd, bucket, block, bits, _ptr(x), _ptr(g)),
           "ring_reduce_scatter")
    return g
