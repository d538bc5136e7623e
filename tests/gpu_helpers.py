"""Shared helpers of the GPU parity tests: library loading, seeded inputs,
oracle comparisons at the benchmark spec's tolerances."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

# tolerances of the parity bar
GRAD_RTOL = 1e-6       # reduced gradient: |d| <= 1e-6 * max|ref| over the block
ADAM_RTOL = 1e-5       # fp32 master, m, v
BF16_ULP = 1           # 16-bit parameter write-back


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def zpp():
    """The CUDA library, built in-tree (raises if it cannot be built)."""
    need_gpu()
    from gradient_comm_codecs_gb300 import _build
    _build.build()
    import gradient_comm_codecs_gb300 as Z
    return Z


def u16(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_to_u16(t)


def np_bytes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint8)


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.float32, copy=False)


def assert_bytes_equal(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:5]}: " \
                          f"got {got[bad[:5]]} want {want[bad[:5]]}"


def assert_f32_bitexact(got, want, what):
    got = np.ascontiguousarray(got, dtype=np.float32)
    want = np.ascontiguousarray(want, dtype=np.float32)
    assert_bytes_equal(got.view(np.uint32), want.view(np.uint32), what)


def assert_grad_close(got, want, block, what):
    """Reduced gradient: within 1e-6 of the block's largest magnitude."""
    got = np.asarray(got, np.float64).reshape(-1, block)
    want = np.asarray(want, np.float64).reshape(-1, block)
    tol = GRAD_RTOL * np.abs(want).max(axis=1, keepdims=True)
    assert np.all(np.abs(got - want) <= tol), what


def assert_rel_close(got, want, rtol, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    ok = np.abs(got - want) <= rtol * np.abs(want) + 1e-30
    assert ok.all(), f"{what}: {np.count_nonzero(~ok)} outside {rtol} relative"


def assert_bf16_ulp(got_u16, want_u16, what, ulp=BF16_ULP):
    # monotone integer image of bf16 bit patterns
    def key(u):
        u = np.asarray(u, np.uint16).astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), u + 0x8000)
    d = np.abs(key(got_u16) - key(want_u16))
    assert d.max(initial=0) <= ulp, f"{what}: max {d.max()} ulp"


def gen_bf16(recipe, seed, stream, n, device="cpu"):
    return synth.fill(recipe, seed, stream, 0, n, device=device)


def grads_for(qgz: W.QgZ, seed, device="cpu", microbatch=0, out=None):
    """[N_d * bucket] bf16: rank r's bucket from grad_stream(r, microbatch)."""
    if out is None:
        out = torch.empty(qgz.nd * qgz.bucket, dtype=torch.bfloat16, device=device)
    for r in range(qgz.nd):
        synth.fill(qgz.grad, seed, synth.grad_stream(r, microbatch), 0, qgz.bucket,
                   out=out[r * qgz.bucket:(r + 1) * qgz.bucket])
    return out
