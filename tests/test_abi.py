"""C-ABI checks that need no GPU: the library builds, loads and exports every
symbol include/zpp.h declares; host-only helpers; argument validation (which
returns before anything touches the device)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gradient_comm_codecs_gb300 import _build, _lib
    _build.build()
    return _lib._lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "zpp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zpp_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ("zpp_qwz_quant", "zpp_qwz_dequant", "zpp_qgz_reorder_quant",
                 "zpp_qgz_hop_reduce", "zpp_shard_adam_step"):
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    from gradient_comm_codecs_gb300 import EXPORTS
    fns = header_functions()
    assert sorted(EXPORTS) == fns
    for name in fns:
        assert hasattr(lib, name), name
    # the binding refers to nothing the header does not declare
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = set(re.findall(r"\bT (zpp_[a-z0-9_]+)\b", out))
    assert set(fns) <= exported


def test_size_helpers(lib):
    import gradient_comm_codecs_gb300 as Z
    import oracle
    for n in (0, 1, 2, 7, 255, 256, 257, 10 ** 9 + 3):
        for bits in (4, 8):
            if bits == 4 and n % 2:
                continue
            assert Z.zpp_codes_bytes(n, bits) == oracle.codes_bytes(n, bits)
        for block in (64, 256, 4096):
            assert Z.zpp_num_blocks(n, block) == oracle.num_blocks(n, block)
    assert Z.zpp_codes_bytes(-1, 8) == -1 and Z.zpp_codes_bytes(10, 3) == -1
    assert Z.zpp_num_blocks(10, 0) == -1


def test_slice_perm_matches_oracle(lib):
    import gradient_comm_codecs_gb300 as Z
    import oracle
    for N in range(1, 9):
        for G in range(1, 9):
            assert Z.zpp_qgz_slice_perm(N, G) == list(oracle.qgz_slice_perm(N, G))
    with pytest.raises(Z.ZppError):
        Z.zpp_qgz_slice_perm(0, 4)


def test_status_strings_and_version(lib):
    import gradient_comm_codecs_gb300 as Z
    assert Z.zpp_status_string(0) == "ok"
    assert "aligned" in Z.zpp_status_string(2)
    assert Z.zpp_abi_version() >> 16 == 1
    assert lib.zpp_last_cuda_error() == b""


A = 1 << 20          # a fake, 16-byte aligned "device pointer" value: never dereferenced
M = A + 8            # misaligned


def test_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    E_ARG, E_MIS = 1, 2
    # qwZ
    assert lib.zpp_qwz_quant(P(A), 4, 256, 256, 3, P(A), P(A), None) == E_ARG     # bits
    assert lib.zpp_qwz_quant(P(A), 4, 256, 100, 8, P(A), P(A), None) == E_ARG     # block not pow2
    assert lib.zpp_qwz_quant(P(A), 4, 256, 32, 8, P(A), P(A), None) == E_ARG      # block < 64
    assert lib.zpp_qwz_quant(P(A), 4, 256, 8192, 8, P(A), P(A), None) == E_ARG    # block > 4096
    assert lib.zpp_qwz_quant(P(A), 4, 255, 256, 4, P(A), P(A), None) == E_ARG     # odd int4 shard
    assert lib.zpp_qwz_quant(P(A), -1, 256, 256, 8, P(A), P(A), None) == E_ARG
    assert lib.zpp_qwz_quant(None, 4, 256, 256, 8, P(A), P(A), None) == E_ARG
    assert lib.zpp_qwz_quant(P(M), 4, 256, 256, 8, P(A), P(A), None) == E_MIS
    assert lib.zpp_qwz_quant(P(A), 4, 256, 256, 8, P(M), P(A), None) == E_MIS
    assert lib.zpp_qwz_quant(None, 0, 256, 256, 8, None, None, None) == 0         # empty: no-op
    assert lib.zpp_qwz_quant(None, 4, 0, 256, 8, None, None, None) == 0
    assert lib.zpp_qwz_dequant(P(A), P(A), 4, 256, 256, 8, P(M), None) == E_MIS
    assert lib.zpp_qwz_dequant(P(A), P(A), 4, 3, 256, 4, P(A), None) == E_ARG
    # qgZ reorder
    assert lib.zpp_qgz_reorder_quant(P(A), 2, 2, 4 * 256 + 4, 256, 4, P(A), P(A), None) == E_ARG
    assert lib.zpp_qgz_reorder_quant(P(A), 0, 2, 4096, 256, 4, P(A), P(A), None) == E_ARG
    assert lib.zpp_qgz_reorder_quant(P(A), 2, 2, 4096, 256, 5, P(A), P(A), None) == E_ARG
    assert lib.zpp_qgz_reorder_quant(P(M), 2, 2, 4096, 256, 4, P(A), P(A), None) == E_MIS
    assert lib.zpp_qgz_reorder_quant(None, 2, 2, 0, 256, 4, None, None, None) == 0


def test_hop_validation(lib):
    from gradient_comm_codecs_gb300._lib import zpp_adam_hparams, zpp_adam_state
    P = ctypes.c_void_p
    hp = zpp_adam_hparams(1e-4, 0.9, 0.999, 1e-8, 1)
    bad_hp = zpp_adam_hparams(1e-4, 0.9, 0.999, 1e-8, 0)
    st = zpp_adam_state(A, A, A, A)
    st_mis = zpp_adam_state(A, M, A, A)
    st_null = zpp_adam_state(A, None, A, A)
    f = lib.zpp_qgz_hop_reduce
    b = 4 * 256 * 4
    ref = ctypes.byref
    # hop 2 with one node: hop 1 is final
    assert f(2, P(A), P(A), 1, 4, b, 256, 4, None, None, P(A), None, None, None) == 1
    # hop 3
    assert f(3, P(A), P(A), 2, 2, b, 256, 4, P(A), P(A), None, None, None, None) == 1
    # non-final hop: needs codes_out and scales_out, and nothing final
    assert f(1, P(A), P(A), 2, 2, b, 256, 4, None, P(A), None, None, None, None) == 1
    assert f(1, P(A), P(A), 2, 2, b, 256, 4, P(A), P(A), P(A), None, None, None) == 1
    assert f(1, P(A), P(A), 2, 2, b, 256, 4, P(A), P(A), None, ref(hp), ref(st), None) == 1
    # final hop: needs grad_out or adam, no codes_out
    assert f(2, P(A), P(A), 2, 2, b, 256, 4, None, None, None, None, None, None) == 1
    assert f(2, P(A), P(A), 2, 2, b, 256, 4, P(A), None, P(A), None, None, None) == 1
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, None, None, ref(hp), None, None) == 1
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, None, None, ref(bad_hp), ref(st), None) == 1
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, None, None, ref(hp), ref(st_null), None) == 1
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, None, None, ref(hp), ref(st_mis), None) == 2
    assert f(2, P(A), P(A), 2, 2, b, 256, 4, None, None, P(M), None, None, None) == 2
    # bucket not a multiple of N_d * block
    assert f(2, P(A), P(A), 2, 2, b + 256, 256, 4, None, None, P(A), None, None, None) == 1
    # empty bucket: valid no-op
    assert f(2, None, None, 2, 2, 0, 256, 4, None, None, P(A), None, None, None) == 0
    # Adam
    g = lib.zpp_shard_adam_step
    assert g(P(A), 100, ref(bad_hp), ref(st), None) == 1
    assert g(P(A), 100, ref(hp), ref(st_null), None) == 1
    assert g(P(M), 100, ref(hp), ref(st), None) == 2
    assert g(P(A), -5, ref(hp), ref(st), None) == 1
    assert g(None, 0, ref(hp), ref(st), None) == 0


def test_binding_rejects_host_tensors():
    import torch
    import gradient_comm_codecs_gb300 as Z
    x = torch.zeros(1024, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        Z.zpp_qwz_quant(x, 1, 1024, 256, 8, x, x, stream=0)


def test_next_rows_validation(lib):
    """The Adam -> qwZ hop, accumulation, hpZ and ring entry points reject bad
    arguments on the host, before anything is enqueued."""
    from gradient_comm_codecs_gb300._lib import zpp_adam_hparams, zpp_adam_state
    P = ctypes.c_void_p
    ref = ctypes.byref
    hp = zpp_adam_hparams(1e-4, 0.9, 0.999, 1e-8, 1)
    st = zpp_adam_state(A, A, A, A)
    # Adam -> qwZ fused final hop
    f = lib.zpp_qgz_final_hop_adam_qwz
    b = 4 * 512
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, None, ref(st), 8, P(A), P(A), None) == 1
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, ref(hp), None, 8, P(A), P(A), None) == 1
    assert f(1, P(A), P(A), 2, 2, b, 256, 4, None, ref(hp), ref(st), 8, P(A), P(A), None) == 1
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, ref(hp), ref(st), 4, P(A), P(A), None) == 3
    assert f(1, P(A), P(A), 1, 4, 4 * 768, 256, 4, None, ref(hp), ref(st), 8, P(A), P(A),
             None) == 3                                             # L = 768: not a multiple of 512
    assert f(1, P(A), P(A), 1, 4, b, 256, 4, None, ref(hp), ref(st), 8, P(M), P(A), None) == 2
    # gradient accumulation
    g = lib.zpp_grad_accumulate
    assert g(P(A), P(A), 100, 2, None) == 1
    assert g(P(A), P(A), -1, 1, None) == 1
    assert g(None, P(A), 100, 1, None) == 1
    assert g(P(A), P(M), 100, 1, None) == 2
    assert g(None, None, 0, 1, None) == 0
    r = lib.zpp_qgz_reorder_quant_acc
    assert r(P(A), P(A), 2, 2, 4 * 256 + 4, 256, 4, P(A), P(A), None) == 1
    assert r(P(A), None, 2, 2, 4096, 256, 4, P(A), P(A), None) == 1
    assert r(P(A), P(M), 2, 2, 4096, 256, 4, P(A), P(A), None) == 2
    assert r(None, None, 2, 2, 0, 256, 4, None, None, None) == 0
    # hpZ
    two = (ctypes.c_void_p * 2)(A, A)
    mis = (ctypes.c_void_p * 2)(A, M)
    h = lib.zpp_hpz_gather
    C = lambda arr: ctypes.cast(arr, ctypes.c_void_p)   # noqa: E731
    assert h(0, 1, 4096, 256, 8, C(two), C(two), P(A), None) == 1
    assert h(65, 1, 4096, 256, 8, C(two), C(two), P(A), None) == 1
    assert h(2, 0, 4096, 256, 8, C(two), C(two), P(A), None) == 1
    assert h(2, 1, 4096, 100, 8, C(two), C(two), P(A), None) == 1
    assert h(2, 1, 4095, 256, 4, C(two), C(two), P(A), None) == 1
    assert h(2, 1, 4096, 256, 8, C(two), None, P(A), None) == 1
    assert h(2, 1, 4096, 256, 8, C(mis), C(two), P(A), None) == 2
    assert h(2, 1, 4096, 256, 8, C(two), C(two), P(M), None) == 2
    assert h(2, 1, 0, 256, 8, None, None, None, None) == 0
    assert lib.zpp_hpz_secondary_bytes(2, 4096, 256, 8) == 2 * (4096 + 4 * 16)
    assert lib.zpp_hpz_secondary_bytes(2, 4096, 256, 4) == 2 * (2048 + 4 * 16)
    assert lib.zpp_hpz_secondary_bytes(2, 4096, 256, 16) == 2 * 2 * 4096
    assert lib.zpp_hpz_secondary_bytes(2, 4096, 256, 5) == -1
    assert lib.zpp_hpz_secondary_bytes(0, 4096, 256, 8) == -1
    # ring
    q = lib.zpp_ring_rs_step
    bb = 4 * 256
    assert q(4, 4, bb, 64, 8, P(A), P(A), P(A), P(A), P(A), P(A), None) == 1    # step >= N_d
    assert q(-1, 4, bb, 64, 8, P(A), P(A), P(A), P(A), P(A), P(A), None) == 1
    assert q(1, 4, bb + 64, 64, 8, P(A), P(A), P(A), P(A), P(A), P(A), None) == 1
    assert q(1, 4, bb, 64, 8, P(A), None, P(A), P(A), P(A), None, None) == 1    # middle: input
    assert q(0, 4, bb, 64, 8, P(A), None, None, None, P(A), None, None) == 1    # first: output
    assert q(3, 4, bb, 64, 8, P(A), P(A), P(A), None, None, None, None) == 1    # last: gradient
    assert q(3, 4, bb, 64, 8, P(A), P(A), P(A), None, None, P(M), None) == 2
    assert q(0, 4, 0, 64, 8, None, None, None, None, None, None, None) == 0


# ---- the binding's size checks (no GPU: they run before any pointer is taken) ----------

def _small_cases():
    import torch
    u16 = lambda n: torch.empty(n, dtype=torch.bfloat16)
    u8 = lambda n: torch.empty(n, dtype=torch.uint8)
    f32 = lambda n: torch.empty(n, dtype=torch.float32)
    import gradient_comm_codecs_gb300 as Z
    n, B = 4 * 1024, 256
    nd, L = 4, 1024                       # 2 nodes x 2, bucket 4096
    cb1, nb1 = nd * (4096 * 4) // 8, nd * 4096 // B
    cb2, nb2 = nd * (2 * L * 4) // 8, nd * 2 * L // B
    st = lambda k=0: (f32(4096 - k), f32(4096), f32(4096), u16(4096))
    return [
        ("x_bf16", lambda: Z.zpp_qwz_quant(u16(2 * n - 1), 2, n, B, 8, u8(2 * n), f32(2 * n // B))),
        ("codes", lambda: Z.zpp_qwz_quant(u16(2 * n), 2, n, B, 8, u8(2 * n - 1), f32(2 * n // B))),
        ("scales", lambda: Z.zpp_qwz_quant(u16(2 * n), 2, n, B, 4, u8(n), f32(2 * n // B - 1))),
        ("y_bf16", lambda: Z.zpp_qwz_dequant(u8(2 * n), f32(2 * n // B), 2, n, B, 8, u16(n))),
        ("grads_bf16", lambda: Z.zpp_qgz_reorder_quant(u16(nd * 4096 - 8), 2, 2, 4096, B, 4,
                                                       u8(cb1), f32(nb1))),
        ("codes", lambda: Z.zpp_qgz_reorder_quant(u16(nd * 4096), 2, 2, 4096, B, 4, u8(cb1 - 1),
                                                  f32(nb1))),
        ("acc", lambda: Z.zpp_qgz_reorder_quant_acc(u16(nd * 4096), f32(nd * 4096 - 1), 2, 2, 4096,
                                                    B, 4, u8(cb1), f32(nb1))),
        ("acc", lambda: Z.zpp_grad_accumulate(u16(100), f32(99), 100, 1)),
        ("codes_in", lambda: Z.zpp_qgz_hop_reduce(1, u8(cb1 - 16), f32(nb1), 2, 2, 4096, B, 4,
                                                  u8(cb2), f32(nb2))),
        ("codes_out", lambda: Z.zpp_qgz_hop_reduce(1, u8(cb1), f32(nb1), 2, 2, 4096, B, 4,
                                                   u8(cb2 - 1), f32(nb2))),
        ("scales_in", lambda: Z.zpp_qgz_hop_reduce(2, u8(cb2), f32(nb2 - 1), 2, 2, 4096, B, 4,
                                                   grad_out=f32(4096))),
        ("grad_out", lambda: Z.zpp_qgz_hop_reduce(2, u8(cb2), f32(nb2), 2, 2, 4096, B, 4,
                                                  grad_out=f32(4095))),
        ("master", lambda: Z.zpp_qgz_hop_reduce(2, u8(cb2), f32(nb2), 2, 2, 4096, B, 4,
                                                adam=(1e-4, .9, .999, 1e-8, 1), state=st(1))),
        ("qwz_codes", lambda: Z.zpp_qgz_final_hop_adam_qwz(2, u8(cb2), f32(nb2), 2, 2, 4096, B, 4,
                                                           None, (1e-4, .9, .999, 1e-8, 1), st(),
                                                           8, u8(4095), f32(4096 // B))),
        ("grads_bf16", lambda: Z.zpp_ring_rs_step(0, 4, 4096, B, 4, u16(4 * 4096 - 1),
                                                  codes_out=u8(4 * 512), scales_out=f32(16))),
        ("codes_out", lambda: Z.zpp_ring_rs_step(0, 4, 4096, B, 4, u16(4 * 4096),
                                                 codes_out=u8(4 * 512 - 1), scales_out=f32(16))),
        ("sec_codes[1]", lambda: Z.zpp_hpz_gather(2, 2, 1024, B, 8, [u8(2048), u8(2047)],
                                                  [f32(8), f32(8)], u16(4096))),
        ("y_bf16", lambda: Z.zpp_hpz_gather(2, 2, 1024, B, 8, [u8(2048), u8(2048)],
                                            [f32(8), f32(8)], u16(4095))),
        ("grad", lambda: Z.zpp_shard_adam_step(f32(99), 100, (1e-4, .9, .999, 1e-8, 1),
                                               (f32(100), f32(100), f32(100), u16(100)))),
        ("param_bf16", lambda: Z.zpp_shard_adam_step(f32(100), 100, (1e-4, .9, .999, 1e-8, 1),
                                                     (f32(100), f32(100), f32(100), u16(99)))),
    ]


@pytest.mark.parametrize("i", range(20))
def test_binding_rejects_undersized_tensors(i):
    """An under-sized tensor raises ValueError naming it before any pointer is
    taken or any call is made."""
    name, call = _small_cases()[i]
    with pytest.raises(ValueError, match=re.escape(name) + " is too small"):
        call()


def test_binding_size_check_accepts_exact_sizes():
    """Exactly sized host tensors pass the size check and stop at the device
    check (nothing reaches the library without a CUDA tensor)."""
    import torch
    import gradient_comm_codecs_gb300 as Z
    n, B = 4096, 256
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        Z.zpp_qwz_quant(torch.empty(2 * n, dtype=torch.bfloat16), 2, n, B, 4,
                        torch.empty(n, dtype=torch.uint8), torch.empty(2 * n // B))
