"""Seeded, counter-based synthetic inputs for the ZeRO++ codec path.

This module is the one thing the CUDA-path tests, the bench and the oracle
tests share.  It holds none of the codec or optimizer arithmetic: it only turns
``(seed, stream, element index)`` into bf16 values drawn from a tabulated
distribution, and it gives bit-identical values on the CPU and on a CUDA
device, so a test can generate a full-size tensor on the GPU and regenerate any
sampled element on the host.

Generator
---------
* Counter hash: ``lowbias32`` (C. Wellons, "Prospecting for Hash Functions",
  2018): ``x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b;
  x ^= x>>16`` on 32-bit words.  Element index ``i`` (64-bit) is hashed as
  ``h = H(H(lo(i) ^ k1) ^ (hi(i) + k2))`` with ``k1, k2`` derived from
  ``(seed, stream)``.  Every step is done in int64 tensors whose values stay
  below 2**49, so no overflow happens on either device (the 32x32-bit products
  are split into 16-bit halves).
* Value: the top 20 bits of ``h`` index a table of 2**20 quantiles
  ``F^-1((j + 0.5) / 2**20)`` of the target distribution, computed in float64
  on the host and rounded to bf16.  There is no transcendental math on the
  device, so host and device agree bit for bit.  Tails are therefore cut at
  the 1 - 2**-21 quantile (|z| <= 4.90 for a normal, |t| <= 132.2 for
  Student-t with 3 degrees of freedom).
* Outliers (two-hop bucket workload): each block of ``outlier_block``
  elements is picked independently with probability ``outlier_prob`` by a
  hash of its global block index; in a picked block one element, also chosen
  by hash, is multiplied by ``outlier_factor`` in fp32 and rounded back to
  bf16 (round to nearest even).

Two implementations of the same function: the tensor path below (any torch
device; what the GPU tests and the bench fill device buffers with) and, on the
host, ``_gen.c`` (plain C, 32-bit unsigned arithmetic, built with gcc on first
use), which the CPU calls of ``fill``/``at`` and ``fill_u16``/``at_u16`` use
when it builds.  The CPU test suite checks that the two agree bit for bit.
"""
from __future__ import annotations

from dataclasses import dataclass
from functools import lru_cache

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

__all__ = [
    "Dist", "Recipe", "WEIGHTS", "MOMENT_M", "MOMENT_V", "SHARD_GRAD", "grad_stream",
    "fill", "at", "fill_u16", "at_u16", "hash32_int", "bf16_to_u16", "u16_to_bf16", "build",
]

_M32 = 0xFFFFFFFF
TABLE_BITS = 20

# stream ids
WEIGHTS = 1
MOMENT_M = 2
MOMENT_V = 3
SHARD_GRAD = 4   # gradients of an owned shard outside the reduced bucket
_OUTLIER_SALT = 0x0D15EA5E


def grad_stream(rank: int, microbatch: int = 0) -> int:
    """Stream id of simulated data-parallel rank ``rank``'s gradient bucket
    (of micro-batch ``microbatch`` when gradients are accumulated)."""
    return 0x1000 + int(rank) + (int(microbatch) << 20)


def hash32_int(x: int) -> int:
    """lowbias32 on a Python int (used for keys)."""
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    x ^= x >> 16
    return x


def _mul32_(x: torch.Tensor, c: int) -> torch.Tensor:
    """x <- (x * c) mod 2**32 in place, for int64 x in [0, 2**32)."""
    hi = x * (c >> 16)
    hi &= 0xFFFF
    hi <<= 16
    x *= c & 0xFFFF
    x += hi
    x &= _M32
    return x


def _hash32_(x: torch.Tensor) -> torch.Tensor:
    x ^= x >> 16
    _mul32_(x, 0x7FEB352D)
    x ^= x >> 15
    _mul32_(x, 0x846CA68B)
    x ^= x >> 16
    return x


def _keys(seed: int, stream: int) -> tuple[int, int]:
    k1 = hash32_int((seed * 0x9E3779B9 + stream * 0x85EBCA6B + 0x632BE5AB) & _M32)
    k2 = hash32_int(k1 ^ 0x5BD1E995)
    return k1, k2


def _hash_index(idx: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """32-bit hash of each int64 element index (new tensor)."""
    k1, k2 = _keys(seed, stream)
    x = idx & _M32
    x ^= k1
    _hash32_(x)
    hi = idx >> 32
    hi += k2
    hi &= _M32
    x ^= hi
    return _hash32_(x)


@dataclass(frozen=True)
class Dist:
    """A tabulated distribution: kind in {"normal", "student_t", "halfnormal"}."""
    kind: str
    scale: float
    dof: float = 0.0


@lru_cache(maxsize=None)
def _table_cpu(dist: Dist) -> torch.Tensor:
    import scipy.special as sp
    import scipy.stats as st
    p = (np.arange(1 << TABLE_BITS, dtype=np.float64) + 0.5) / float(1 << TABLE_BITS)
    if dist.kind == "normal":
        q = sp.ndtri(p)
    elif dist.kind == "student_t":
        q = st.t.ppf(p, dist.dof)
    elif dist.kind == "halfnormal":
        q = sp.ndtri(0.5 + 0.5 * p)
    else:
        raise ValueError(f"unknown distribution {dist.kind!r}")
    q = (q * dist.scale).astype(np.float32)
    return torch.from_numpy(q).to(torch.bfloat16)


_table_dev: dict = {}


def _table(dist: Dist, device: torch.device) -> torch.Tensor:
    device = torch.device(device)
    if device.type == "cpu":
        return _table_cpu(dist)
    key = (dist, str(device))
    t = _table_dev.get(key)
    if t is None:
        t = _table_cpu(dist).to(device)
        _table_dev[key] = t
    return t


@dataclass(frozen=True)
class Recipe:
    """How one tensor of a workload is drawn."""
    dist: Dist
    outlier_block: int = 0          # 0: no outliers
    outlier_prob: float = 0.0
    outlier_factor: float = 1.0


def _values_at(recipe: Recipe, seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    h = _hash_index(idx, seed, stream)
    h >>= 32 - TABLE_BITS
    out = _table(recipe.dist, idx.device)[h]
    del h
    if recipe.outlier_block:
        B = int(recipe.outlier_block)
        thr = int(recipe.outlier_prob * 4294967296.0)
        blk = idx // B
        pick = _hash_index(blk, seed, stream ^ _OUTLIER_SALT)
        sel = pick < thr
        elem = _hash_index(blk, seed, stream ^ (_OUTLIER_SALT + 1)) % B
        sel &= elem == (idx - blk * B)
        if bool(sel.any()):
            boosted = (out[sel].float() * float(recipe.outlier_factor)).to(torch.bfloat16)
            out[sel] = boosted
    return out


def _fill_torch(recipe: Recipe, seed: int, stream: int, start: int, count: int,
                out: torch.Tensor, chunk: int) -> torch.Tensor:
    for c0 in range(0, count, chunk):
        c1 = min(count, c0 + chunk)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=out.device)
        out[c0:c1] = _values_at(recipe, seed, stream, idx)
        del idx
    return out


def fill(recipe: Recipe, seed: int, stream: int, start: int, count: int,
         device="cpu", out: torch.Tensor | None = None, chunk: int = 1 << 25) -> torch.Tensor:
    """bf16 values of global indices [start, start+count) of ``stream``."""
    device = torch.device(device) if out is None else out.device
    if out is None:
        out = torch.empty(count, dtype=torch.bfloat16, device=device)
    assert out.numel() == count and out.dtype == torch.bfloat16
    if device.type == "cpu" and out.is_contiguous() and _host_lib() is not None:
        fill_u16(recipe, seed, stream, start, count, out=out.view(torch.int16).numpy().view(np.uint16))
        return out
    return _fill_torch(recipe, seed, stream, start, count, out, chunk)


def at(recipe: Recipe, seed: int, stream: int, idx) -> torch.Tensor:
    """bf16 values at arbitrary global indices (CPU unless idx is on a device)."""
    if not isinstance(idx, torch.Tensor):
        if _host_lib() is not None:
            return u16_to_bf16(at_u16(recipe, seed, stream, idx))
        idx = torch.as_tensor(np.asarray(idx, dtype=np.int64))
    return _values_at(recipe, seed, stream, idx.to(torch.int64).reshape(-1).clone())


# ---- host fast path (_gen.c) ---------------------------------------------------------

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "_gen.c")
_SO = os.path.join(_HERE, "libsynth.so")
_build_lock = threading.Lock()
_lib = None
_lib_failed = False


class _Outliers(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int64), ("thr", ctypes.c_uint64), ("p1", ctypes.c_uint32),
                ("p2", ctypes.c_uint32), ("e1", ctypes.c_uint32), ("e2", ctypes.c_uint32),
                ("factor", ctypes.c_float)]


def build(force: bool = False) -> str:
    """Compile the host generator with gcc, in-tree next to its source."""
    with _build_lock:
        if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
            tmp = _SO + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall",
                                   _SRC, "-o", tmp])
            os.replace(tmp, _SO)
    return _SO


def _host_lib():
    """The compiled host generator, or None when gcc is unavailable (the
    tensor path then serves the host too)."""
    global _lib, _lib_failed
    if _lib is not None or _lib_failed:
        return _lib
    try:
        build()
        try:
            lib = ctypes.CDLL(_SO)
        except OSError:  # e.g. a binary built for another machine
            build(force=True)
            lib = ctypes.CDLL(_SO)
    except (OSError, subprocess.CalledProcessError):
        _lib_failed = True
        return None
    P, I64, I32, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    for name in ("synth_fill", "synth_at"):
        fn = getattr(lib, name)
        fn.restype = None
    lib.synth_fill.argtypes = [P, P, I32, U32, U32, I64, I64, ctypes.POINTER(_Outliers)]
    lib.synth_at.argtypes = [P, P, I32, U32, U32, P, I64, ctypes.POINTER(_Outliers)]
    _lib = lib
    return lib


@lru_cache(maxsize=None)
def _table_u16(dist: Dist) -> np.ndarray:
    return np.ascontiguousarray(bf16_to_u16(_table_cpu(dist)))


def _outliers(recipe: Recipe, seed: int, stream: int):
    if not recipe.outlier_block:
        return None
    p1, p2 = _keys(seed, stream ^ _OUTLIER_SALT)
    e1, e2 = _keys(seed, stream ^ (_OUTLIER_SALT + 1))
    return _Outliers(int(recipe.outlier_block), int(recipe.outlier_prob * 4294967296.0),
                     p1, p2, e1, e2, float(recipe.outlier_factor))


def fill_u16(recipe: Recipe, seed: int, stream: int, start: int, count: int,
             out: np.ndarray | None = None) -> np.ndarray:
    """Host bf16 bit patterns (uint16) of global indices [start, start+count)."""
    lib = _host_lib()
    if out is None:
        out = np.empty(int(count), np.uint16)
    assert out.dtype == np.uint16 and out.size == count and out.flags.c_contiguous
    if lib is None:
        out[:] = bf16_to_u16(_fill_torch(recipe, seed, stream, start, count,
                                         torch.empty(count, dtype=torch.bfloat16), 1 << 22))
        return out
    k1, k2 = _keys(seed, stream)
    o = _outliers(recipe, seed, stream)
    tab = _table_u16(recipe.dist)
    lib.synth_fill(out.ctypes.data, tab.ctypes.data, 32 - TABLE_BITS, k1, k2, int(start),
                   int(count), ctypes.byref(o) if o is not None else None)
    return out


def at_u16(recipe: Recipe, seed: int, stream: int, idx) -> np.ndarray:
    """Host bf16 bit patterns (uint16) at arbitrary global indices."""
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1))
    lib = _host_lib()
    if lib is None:
        return bf16_to_u16(_values_at(recipe, seed, stream, torch.from_numpy(idx.copy())))
    out = np.empty(idx.size, np.uint16)
    k1, k2 = _keys(seed, stream)
    o = _outliers(recipe, seed, stream)
    tab = _table_u16(recipe.dist)
    lib.synth_at(out.ctypes.data, tab.ctypes.data, 32 - TABLE_BITS, k1, k2, idx.ctypes.data,
                 idx.size, ctypes.byref(o) if o is not None else None)
    return out


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a bf16 tensor as a numpy uint16 array (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u16_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
