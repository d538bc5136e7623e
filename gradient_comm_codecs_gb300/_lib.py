"""ctypes binding of libzpp.so: the C ABI of include/zpp.h, one Python function
per entry point with the same name.  Argument marshalling only -- every step
of the path runs in the CUDA kernels behind these calls.

Tensors are passed as torch tensors on a CUDA device (contiguous, of the dtype
the header states) and turned into raw device pointers; `stream` defaults to
torch's current stream on the tensors' device, and the call runs with that
device current.  Before the C call every tensor argument is checked against
the bytes the call will read or write (computed from the scalar arguments by
the header's size rules) and against the other tensors' device: a tensor that
is too small, or on another device, raises ValueError and nothing is
launched.  (Raw integer pointers are passed through unchecked.)  A nonzero
status raises ``ZppError``.  If the library has not been built the first call
raises: there is no fallback path.
"""
from __future__ import annotations

import contextlib
import ctypes
import numbers
import os

import torch

from ._build import LIB

ZPP_OK, ZPP_ERR_INVALID_ARG, ZPP_ERR_MISALIGNED, ZPP_ERR_UNSUPPORTED, ZPP_ERR_CUDA = range(5)

# every symbol include/zpp.h declares
EXPORTS = (
    "zpp_qwz_quant", "zpp_qwz_dequant", "zpp_qgz_reorder_quant", "zpp_grad_accumulate",
    "zpp_qgz_reorder_quant_acc", "zpp_qgz_hop_reduce", "zpp_qgz_final_hop_adam_qwz",
    "zpp_hpz_gather", "zpp_hpz_secondary_bytes", "zpp_ring_rs_step", "zpp_shard_adam_step", "zpp_codes_bytes", "zpp_num_blocks", "zpp_qgz_slice_perm",
    "zpp_status_string", "zpp_last_cuda_error", "zpp_abi_version",
)


class ZppError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib().zpp_status_string(status).decode()
        if status == ZPP_ERR_CUDA:
            msg += ": " + _lib().zpp_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")


class zpp_adam_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("step", ctypes.c_int32)]


class zpp_adam_state(ctypes.Structure):
    _fields_ = [("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("param_bf16", ctypes.c_void_p)]


_handle = None


def library_path() -> str:
    return LIB


def _lib():
    global _handle
    if _handle is not None:
        return _handle
    if not os.path.exists(LIB):
        raise RuntimeError(
            f"{LIB} is not built: run `python -m gradient_comm_codecs_gb300._build` "
            "(or __graft_entry__.build()) first; there is no fallback implementation")
    lib = ctypes.CDLL(LIB)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    HP, ST = ctypes.POINTER(zpp_adam_hparams), ctypes.POINTER(zpp_adam_state)
    sigs = {
        "zpp_qwz_quant": (I32, [P, I64, I64, I32, I32, P, P, P]),
        "zpp_qwz_dequant": (I32, [P, P, I64, I64, I32, I32, P, P]),
        "zpp_qgz_reorder_quant": (I32, [P, I32, I32, I64, I32, I32, P, P, P]),
        "zpp_grad_accumulate": (I32, [P, P, I64, I32, P]),
        "zpp_qgz_reorder_quant_acc": (I32, [P, P, I32, I32, I64, I32, I32, P, P, P]),
        "zpp_qgz_hop_reduce": (I32, [I32, P, P, I32, I32, I64, I32, I32, P, P, P, HP, ST, P]),
        "zpp_qgz_final_hop_adam_qwz": (I32, [I32, P, P, I32, I32, I64, I32, I32, P, HP, ST, I32, P,
                                              P, P]),
        "zpp_ring_rs_step": (I32, [I32, I32, I64, I32, I32, P, P, P, P, P, P, P]),
        "zpp_hpz_gather": (I32, [I32, I32, I64, I32, I32, P, P, P, P]),
        "zpp_hpz_secondary_bytes": (I64, [I32, I64, I32, I32]),
        "zpp_shard_adam_step": (I32, [P, I64, HP, ST, P]),
        "zpp_codes_bytes": (I64, [I64, I32]),
        "zpp_num_blocks": (I64, [I64, I32]),
        "zpp_qgz_slice_perm": (I32, [I32, I32, P]),
        "zpp_status_string": (ctypes.c_char_p, [I32]),
        "zpp_last_cuda_error": (ctypes.c_char_p, []),
        "zpp_abi_version": (I32, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _handle = lib
    return lib


# ---- marshalling helpers ----------------------------------------------------------

def _dev(t, dtype, name):
    """Raw device pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):  # already a raw device pointer
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor or a device pointer")
    if not t.is_cuda:
        raise ValueError(f"{name}: tensor must be on a CUDA device")
    if dtype is not None and t.dtype not in dtype:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    return t.data_ptr()


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (
    torch.bfloat16, torch.int16)
_BYTES = (torch.uint8, torch.int8)
_F32 = (torch.float32,)


def _stream(stream, *tensors):
    if stream is None:
        dev = next((t.device for t in tensors if isinstance(t, torch.Tensor)), None)
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status, where):
    if status != ZPP_OK:
        raise ZppError(status, where)


# ---- size and device checks (before anything is launched) ----------------------------

def _cb(n, bits):
    """Code bytes of n elements (the header's zpp_codes_bytes rule)."""
    return (n * bits + 7) // 8


def _nb(n, block):
    """Blocks of n elements (the header's zpp_num_blocks rule)."""
    return -(-n // block)


_NULL = contextlib.nullcontext()


def _guard(where, *needs):
    """Check every (tensor, bytes needed, name) of a call and return a context
    that makes the tensors' device current (a no-op context when it already
    is).  Sizes are only checked when the scalar arguments are well formed;
    malformed ones are left for the library's own validation (it returns
    ZPP_ERR_INVALID_ARG)."""
    dev = None
    for t, need, name in needs:
        if t is None or type(t) is int:
            continue
        if not isinstance(t, torch.Tensor):
            continue
        if t.is_cuda:
            if dev is None:
                dev = t.device
            elif t.device != dev:
                raise ValueError(f"{where}: {name} is on {t.device}, other arguments on {dev}")
        if need:
            have = t.numel() * t.element_size()
            if have < need:
                raise ValueError(f"{where}: {name} is too small: {have} bytes, the call "
                                 f"accesses {need}")
    if dev is None or dev.index == torch.cuda.current_device():
        return _NULL
    return torch.cuda.device(dev)


def _ok(*vals):
    """True when every size argument is a non-negative integer."""
    for v in vals:
        if type(v) is not int and not isinstance(v, numbers.Integral):
            return False
        if v < 0:
            return False
    return True


def _codec_ok(block, bits):
    return _ok(block, bits) and block > 0 and bits in (4, 8, 16)


# ---- entry points ---------------------------------------------------------------------

def zpp_qwz_quant(x_bf16, nranks, shard_elems, block, bits, codes, scales, stream=None):
    ok = _ok(nranks, shard_elems) and _codec_ok(block, bits)
    n = nranks * shard_elems if ok else None
    with _guard("zpp_qwz_quant", (x_bf16, ok and 2 * n, "x_bf16"),
                (codes, ok and nranks * _cb(shard_elems, bits), "codes"),
                (scales, ok and 4 * nranks * _nb(shard_elems, block), "scales")):
        _check(_lib().zpp_qwz_quant(_dev(x_bf16, _BF16, "x_bf16"), nranks, shard_elems, block,
                                    bits, _dev(codes, _BYTES, "codes"),
                                    _dev(scales, _F32, "scales"), _stream(stream, x_bf16)),
               "zpp_qwz_quant")


def zpp_qwz_dequant(codes, scales, nranks, shard_elems, block, bits, y_bf16, stream=None):
    ok = _ok(nranks, shard_elems) and _codec_ok(block, bits)
    with _guard("zpp_qwz_dequant", (codes, ok and nranks * _cb(shard_elems, bits), "codes"),
                (scales, ok and 4 * nranks * _nb(shard_elems, block), "scales"),
                (y_bf16, ok and 2 * nranks * shard_elems, "y_bf16")):
        _check(_lib().zpp_qwz_dequant(_dev(codes, _BYTES, "codes"), _dev(scales, _F32, "scales"),
                                      nranks, shard_elems, block, bits,
                                      _dev(y_bf16, _BF16, "y_bf16"), _stream(stream, codes)),
               "zpp_qwz_dequant")


def _qgz_msg(nodes, gpus_per_node, bucket_elems, block, bits):
    """(ranks, one-shot code bytes, one-shot scale bytes) of a qgZ bucket, or
    None when the arguments are malformed."""
    if not (_ok(nodes, gpus_per_node, bucket_elems) and _codec_ok(block, bits)):
        return None
    nd = nodes * gpus_per_node
    if nd < 1:
        return None
    return nd, nd * _cb(bucket_elems, bits), 4 * nd * (bucket_elems // block)


def zpp_qgz_reorder_quant(grads_bf16, nodes, gpus_per_node, bucket_elems, block, bits, codes,
                          scales, stream=None):
    m = _qgz_msg(nodes, gpus_per_node, bucket_elems, block, bits)
    with _guard("zpp_qgz_reorder_quant",
                (grads_bf16, m and 2 * m[0] * bucket_elems, "grads_bf16"),
                (codes, m and m[1], "codes"), (scales, m and m[2], "scales")):
        _check(_lib().zpp_qgz_reorder_quant(_dev(grads_bf16, _BF16, "grads_bf16"), nodes,
                                            gpus_per_node, bucket_elems, block, bits,
                                            _dev(codes, _BYTES, "codes"),
                                            _dev(scales, _F32, "scales"),
                                            _stream(stream, grads_bf16)),
               "zpp_qgz_reorder_quant")


def zpp_grad_accumulate(grads_bf16, acc, n, first, stream=None):
    ok = _ok(n)
    with _guard("zpp_grad_accumulate", (grads_bf16, ok and 2 * n, "grads_bf16"),
                (acc, ok and 4 * n, "acc")):
        _check(_lib().zpp_grad_accumulate(_dev(grads_bf16, _BF16, "grads_bf16"),
                                          _dev(acc, _F32, "acc"), n, int(first),
                                          _stream(stream, grads_bf16)),
               "zpp_grad_accumulate")


def zpp_qgz_reorder_quant_acc(grads_bf16, acc, nodes, gpus_per_node, bucket_elems, block, bits,
                              codes, scales, stream=None):
    m = _qgz_msg(nodes, gpus_per_node, bucket_elems, block, bits)
    with _guard("zpp_qgz_reorder_quant_acc",
                (grads_bf16, m and 2 * m[0] * bucket_elems, "grads_bf16"),
                (acc, m and 4 * m[0] * bucket_elems, "acc"),
                (codes, m and m[1], "codes"), (scales, m and m[2], "scales")):
        _check(_lib().zpp_qgz_reorder_quant_acc(_dev(grads_bf16, _BF16, "grads_bf16"),
                                                _dev(acc, _F32, "acc"), nodes, gpus_per_node,
                                                bucket_elems, block, bits,
                                                _dev(codes, _BYTES, "codes"),
                                                _dev(scales, _F32, "scales"),
                                                _stream(stream, grads_bf16)),
               "zpp_qgz_reorder_quant_acc")


def _adam_args(adam, state):
    hp = st = None
    if adam is not None:
        hp = zpp_adam_hparams(*adam) if isinstance(adam, (tuple, list)) else adam
    if state is not None:
        if isinstance(state, (tuple, list)):
            master, m, v, param = state
            st = zpp_adam_state(_dev(master, _F32, "master"), _dev(m, _F32, "m"),
                                _dev(v, _F32, "v"), _dev(param, _BF16, "param_bf16"))
        else:
            st = state
    return (ctypes.byref(hp) if hp is not None else None,
            ctypes.byref(st) if st is not None else None, hp, st)


def _state_needs(state, n):
    """(tensor, bytes, name) of an Adam state tuple over n parameters."""
    if not isinstance(state, (tuple, list)):
        return []
    master, m, v, param = state
    ok = n is not None
    return [(master, ok and 4 * n, "master"), (m, ok and 4 * n, "m"), (v, ok and 4 * n, "v"),
            (param, ok and 2 * n, "param_bf16")]


def _hop_needs(hop, nodes, gpus_per_node, bucket_elems, block, bits, codes_in, scales_in,
               codes_out, scales_out, grad_out, state):
    m = _qgz_msg(nodes, gpus_per_node, bucket_elems, block, bits)
    needs = []
    if m is None or hop not in (1, 2):
        return [(codes_in, None, "codes_in"), (scales_in, None, "scales_in"),
                (codes_out, None, "codes_out"), (scales_out, None, "scales_out"),
                (grad_out, None, "grad_out")] + _state_needs(state, None)
    nd = m[0]
    L = bucket_elems // nd
    two = (nd * _cb(nodes * L, bits), 4 * nd * (nodes * L // block))  # hop-1 message
    cin, sin = (m[1], m[2]) if hop == 1 else two
    needs += [(codes_in, cin, "codes_in"), (scales_in, sin, "scales_in"),
              (codes_out, two[0], "codes_out"), (scales_out, two[1], "scales_out"),
              (grad_out, 4 * bucket_elems, "grad_out")]
    return needs + _state_needs(state, bucket_elems)


def zpp_qgz_hop_reduce(hop, codes_in, scales_in, nodes, gpus_per_node, bucket_elems, block, bits,
                       codes_out=None, scales_out=None, grad_out=None, adam=None, state=None,
                       stream=None):
    """`adam`: (lr, beta1, beta2, eps, step) or zpp_adam_hparams; `state`:
    (master, m, v, param_bf16_or_None) tensors or zpp_adam_state."""
    needs = _hop_needs(hop, nodes, gpus_per_node, bucket_elems, block, bits, codes_in, scales_in,
                       codes_out, scales_out, grad_out, state)
    with _guard("zpp_qgz_hop_reduce", *needs):
        hp, st, _keep1, _keep2 = _adam_args(adam, state)
        _check(_lib().zpp_qgz_hop_reduce(hop, _dev(codes_in, _BYTES, "codes_in"),
                                         _dev(scales_in, _F32, "scales_in"), nodes, gpus_per_node,
                                         bucket_elems, block, bits,
                                         _dev(codes_out, _BYTES, "codes_out"),
                                         _dev(scales_out, _F32, "scales_out"),
                                         _dev(grad_out, _F32, "grad_out"), hp, st,
                                         _stream(stream, codes_in)), "zpp_qgz_hop_reduce")


def zpp_qgz_final_hop_adam_qwz(hop, codes_in, scales_in, nodes, gpus_per_node, bucket_elems,
                               block, bits, grad_out, adam, state, qwz_bits, qwz_codes,
                               qwz_scales, stream=None):
    needs = _hop_needs(hop, nodes, gpus_per_node, bucket_elems, block, bits, codes_in, scales_in,
                       None, None, grad_out, state)
    ok = _ok(bucket_elems) and _codec_ok(block, bits)
    needs += [(qwz_codes, ok and bucket_elems, "qwz_codes"),
              (qwz_scales, ok and 4 * (bucket_elems // block), "qwz_scales")]
    with _guard("zpp_qgz_final_hop_adam_qwz", *needs):
        hp, st, _keep1, _keep2 = _adam_args(adam, state)
        _check(_lib().zpp_qgz_final_hop_adam_qwz(
            hop, _dev(codes_in, _BYTES, "codes_in"), _dev(scales_in, _F32, "scales_in"), nodes,
            gpus_per_node, bucket_elems, block, bits, _dev(grad_out, _F32, "grad_out"), hp, st,
            qwz_bits, _dev(qwz_codes, _BYTES, "qwz_codes"), _dev(qwz_scales, _F32, "qwz_scales"),
            _stream(stream, codes_in)), "zpp_qgz_final_hop_adam_qwz")


def zpp_ring_rs_step(step, nranks, bucket_elems, block, bits, grads_bf16, codes_in=None,
                     scales_in=None, codes_out=None, scales_out=None, grad_out=None, stream=None):
    ok = _ok(nranks, bucket_elems) and nranks > 0 and _codec_ok(block, bits)
    L = bucket_elems // nranks if ok else 0
    cb, sb = (nranks * _cb(L, bits), 4 * nranks * (L // block)) if ok else (None, None)
    with _guard("zpp_ring_rs_step", (grads_bf16, ok and 2 * nranks * bucket_elems, "grads_bf16"),
                (codes_in, cb, "codes_in"), (scales_in, sb, "scales_in"),
                (codes_out, cb, "codes_out"), (scales_out, sb, "scales_out"),
                (grad_out, ok and 4 * bucket_elems, "grad_out")):
        _check(_lib().zpp_ring_rs_step(step, nranks, bucket_elems, block, bits,
                                       _dev(grads_bf16, _BF16, "grads_bf16"),
                                       _dev(codes_in, _BYTES, "codes_in"),
                                       _dev(scales_in, _F32, "scales_in"),
                                       _dev(codes_out, _BYTES, "codes_out"),
                                       _dev(scales_out, _F32, "scales_out"),
                                       _dev(grad_out, _F32, "grad_out"),
                                       _stream(stream, grads_bf16)),
               "zpp_ring_rs_step")


def zpp_hpz_gather(gpus_per_node, shards_per_rank, shard_elems, block, bits, sec_codes,
                   sec_scales, y_bf16, stream=None):
    """`sec_codes`/`sec_scales`: one device tensor (or pointer) per local rank
    (`sec_scales` None for bits 16)."""
    G = len(sec_codes)
    if G != gpus_per_node:
        raise ValueError("one secondary partition per local rank")
    ok = _ok(shards_per_rank, shard_elems) and _codec_ok(block, bits)
    N = shards_per_rank
    cbytes = (N * (2 * shard_elems if bits == 16 else _cb(shard_elems, bits))) if ok else None
    needs = [(t, cbytes, f"sec_codes[{l}]") for l, t in enumerate(sec_codes)]
    if bits != 16:
        if sec_scales is None or len(sec_scales) != G:
            raise ValueError("one scale tensor per local rank")
        needs += [(t, ok and 4 * N * _nb(shard_elems, block), f"sec_scales[{l}]")
                  for l, t in enumerate(sec_scales)]
    needs.append((y_bf16, ok and 2 * G * N * shard_elems, "y_bf16"))
    with _guard("zpp_hpz_gather", *needs):
        cp = (ctypes.c_void_p * G)(*[_dev(t, _BF16 if bits == 16 else _BYTES, "sec_codes")
                                     for t in sec_codes])
        sp = None
        if bits != 16:
            sp = (ctypes.c_void_p * G)(*[_dev(t, _F32, "sec_scales") for t in sec_scales])
        _check(_lib().zpp_hpz_gather(gpus_per_node, shards_per_rank, shard_elems, block, bits,
                                     ctypes.cast(cp, ctypes.c_void_p),
                                     None if sp is None else ctypes.cast(sp, ctypes.c_void_p),
                                     _dev(y_bf16, _BF16, "y_bf16"), _stream(stream, y_bf16)),
               "zpp_hpz_gather")


def zpp_hpz_secondary_bytes(shards_per_rank, shard_elems, block, bits):
    return int(_lib().zpp_hpz_secondary_bytes(shards_per_rank, shard_elems, block, bits))


def zpp_shard_adam_step(grad, n, adam, state, stream=None):
    ok = _ok(n)
    with _guard("zpp_shard_adam_step", (grad, ok and 4 * n, "grad"),
                *_state_needs(state, n if ok else None)):
        hp, st, _keep1, _keep2 = _adam_args(adam, state)
        _check(_lib().zpp_shard_adam_step(_dev(grad, _F32, "grad"), n, hp, st,
                                          _stream(stream, grad)),
               "zpp_shard_adam_step")


def zpp_codes_bytes(n, bits):
    return int(_lib().zpp_codes_bytes(n, bits))


def zpp_num_blocks(n, block):
    return int(_lib().zpp_num_blocks(n, block))


def zpp_qgz_slice_perm(nodes, gpus_per_node):
    arr = (ctypes.c_int32 * (nodes * gpus_per_node))()
    _check(_lib().zpp_qgz_slice_perm(nodes, gpus_per_node, arr), "zpp_qgz_slice_perm")
    return list(arr)


def zpp_status_string(status):
    return _lib().zpp_status_string(status).decode()


def zpp_abi_version():
    return int(_lib().zpp_abi_version())
