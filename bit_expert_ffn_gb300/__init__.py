"""GB300 (sm_103a) routed-expert MoE layer with 2-/3-bit block-quantised experts.

This module is the Python binding of ``libmoe_gb300.so``: every function
named ``moe_*`` here marshals torch tensors into the C call of the same name
declared in ``include/moe_gb300.h`` and raises :class:`MoeError` on a non-OK
status.  All arithmetic runs in the library's CUDA kernels; there is no other
code path, and importing a function of this module without the built library
raises at once.  Tensors are passed by device pointer and work is enqueued on
the current torch CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")
SYNTH_PATH = os.path.join(HERE, "libmoe_synth.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe_gb300.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_NONFINITE, MOE_ERR_BOUNDS = 4, 5, 6, 7
MOE_ERR_RANGE = 8
MOE_ID_NOT_LOCAL = -1
MOE_F32, MOE_BF16 = 0, 1
MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_PREFILL, MOE_PATH_PREFILL_FP8 = 0, 1, 2, 3
RMS_EPS = 1e-6  # normalisation in front of each stacked layer

_lock = threading.Lock()
_lib = None
_synth = None


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class moe_expert_arena(ctypes.Structure):
    _fields_ = [
        ("bits", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("I", ctypes.c_int32),
        ("E", ctypes.c_int32),
        ("gu_codes", ctypes.c_void_p),
        ("gu_scales", ctypes.c_void_p),
        ("d_codes", ctypes.c_void_p),
        ("d_scales", ctypes.c_void_p),
    ]


class moe_layer_weights(ctypes.Structure):
    _fields_ = [
        ("experts", moe_expert_arena),
        ("w_router", ctypes.c_void_p),
        ("bias", ctypes.c_void_p),
        ("shared_wg", ctypes.c_void_p),
        ("shared_wu", ctypes.c_void_p),
        ("shared_wd", ctypes.c_void_p),
        ("shared_I", ctypes.c_int32),
    ]


class moe_decode_options(ctypes.Structure):
    _fields_ = [
        ("route_tail_skip", ctypes.c_int32),
        ("hot_experts", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_PSZ = ctypes.POINTER(ctypes.c_size_t)

# name -> argtypes (restype moe_status = int unless noted)
_SIGS = {
    "moe_check_status": [_P, _I32, _P],
    "moe_packed_size": [_I32, _I64, _I64, _PSZ, _PSZ],
    "moe_pack_experts": [_I32, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P],
    "moe_unpack_experts": [_I32, _I64, _I64, _I64, _P, _P, _P],
    "moe_router_workspace_size": [_I32, _I32, _I32, _I32, _PSZ],
    "moe_router_topk": [_P, _I32, _I32, _P, _P, _I32, _I32, _P, _P, _P, _P, _SZ, _P, _P],
    "moe_topk_from_logits": [_P, _I32, _I32, _I32, _P, _P, _P, _P],
    "moe_permute_workspace_size": [_I32, _I32, _I32, _PSZ],
    "moe_shard_ids": [_P, _I64, _I32, _I32, _P, _P],
    "moe_permute": [_P, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P, _P],
    "moe_permute_noalloc": [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P],
    "moe_expert_forward_workspace_size": [ctypes.POINTER(moe_expert_arena), _I32, _I32, _I32, _PSZ],
    "moe_expert_forward": [ctypes.POINTER(moe_expert_arena), _P, _I32, _P, _P, _I32, _P, _P, _P, _P, _I32, _I32,
                           _I32, _P, _SZ, _P, _P],
    "moe_shared_expert_workspace_size": [_I32, _I32, _I32, _PSZ],
    "moe_shared_expert": [_P, _P, _P, _I32, _I32, _P, _I32, _P, _I32, _I32, _P, _SZ, _P, _P],
    "moe_f32_to_bf16": [_P, _P, _I64, _P],
    "moe_decode_workspace_size": [_I32, _I32, _I32, _I32, _I32, _I32, _PSZ],
    "moe_decode_forward": [ctypes.POINTER(moe_layer_weights), _I32, _P, _I32, _I32, ctypes.c_float, _P, _P, _P, _SZ,
                           _P, _P],
    "moe_decode_forward_ex": [ctypes.POINTER(moe_layer_weights), _I32, _P, _I32, _I32, ctypes.c_float,
                              ctypes.POINTER(moe_decode_options), _P, _P, _P, _SZ, _P, _P],
    "moe_rms_norm_bf16": [_P, _P, _I32, _I32, ctypes.c_float, _P],
    "moe_selftest_barrier": [ctypes.c_uint, _I32, _P, _SZ, _P, _P],
}


def load():
    """Load libmoe_gb300.so (and the input generator library); raise if it is not built."""
    global _lib, _synth
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise MoeError(MOE_ERR_CUDA, f"{LIB_PATH} is not built: run `python -m bit_expert_ffn_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, args in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            L.moe_last_error.restype = ctypes.c_char_p
            L.moe_last_error.argtypes = []
            L.moe_status_name.restype = ctypes.c_char_p
            L.moe_status_name.argtypes = [ctypes.c_int]
            _lib = L
        if _synth is None and os.path.exists(SYNTH_PATH):
            S = ctypes.CDLL(SYNTH_PATH)
            S.moe_synth_codes.argtypes = [ctypes.c_uint64, ctypes.c_uint64, _I64, _I32, _P, _P]
            S.moe_synth_codes.restype = ctypes.c_int
            S.moe_synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, _I64, ctypes.c_float, ctypes.c_float,
                                           _I32, _P, _P]
            S.moe_synth_normal.restype = ctypes.c_int
            _synth = S
    return _lib


def lib():
    return _lib if _lib is not None else load()


def synth_lib():
    load()
    if _synth is None:
        raise MoeError(MOE_ERR_CUDA, f"{SYNTH_PATH} is not built")
    return _synth


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def moe_status_name(s: int) -> str:
    return lib().moe_status_name(int(s)).decode()


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, f"{what}: {moe_last_error()}")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr() if t.numel() else None


def _stream(stream=None):
    """The stream handle: an int, a torch stream, or the current torch stream."""
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    if stream is None:
        import torch

        if not torch.cuda.is_available():  # host-side argument checks still run
            return ctypes.c_void_p(0)
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _size(fn, *args) -> int:
    out = ctypes.c_size_t(0)
    _check(fn(*args, ctypes.byref(out)), fn.__name__)
    return out.value


# ----------------------------------------------------------------- status

def moe_check_status(dev_status, reset=True, stream=None) -> int:
    """Synchronise and read the device status word; returns the status (no raise)."""
    return lib().moe_check_status(_ptr(dev_status), int(reset), _stream(stream))


# ----------------------------------------------------------------- packing

def moe_packed_size(bits: int, rows: int, cols: int):
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().moe_packed_size(bits, rows, cols, ctypes.byref(cb), ctypes.byref(sb)), "moe_packed_size")
    return cb.value, sb.value


def moe_pack_experts(bits, n_mats, rows, cols, codes, scales, packed_codes, packed_scales, dev_status=None,
                     stream=None):
    _check(lib().moe_pack_experts(bits, n_mats, rows, cols, _ptr(codes), _ptr(scales), _ptr(packed_codes),
                                  _ptr(packed_scales), _ptr(dev_status), _stream(stream)), "moe_pack_experts")


def moe_unpack_experts(bits, n_mats, rows, cols, packed_codes, codes, stream=None):
    _check(lib().moe_unpack_experts(bits, n_mats, rows, cols, _ptr(packed_codes), _ptr(codes), _stream(stream)),
           "moe_unpack_experts")


# ----------------------------------------------------------------- router

def moe_router_workspace_size(T, H, E, logits_given):
    return _size(lib().moe_router_workspace_size, T, H, E, int(logits_given))


def moe_router_topk(x_bf16, T, H, w_router, bias, E, k, logits_out, topk_ids, topk_w, ws=None, ws_bytes=0,
                    dev_status=None, stream=None):
    _check(lib().moe_router_topk(_ptr(x_bf16), T, H, _ptr(w_router), _ptr(bias), E, k, _ptr(logits_out),
                                 _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)),
           "moe_router_topk")


def moe_topk_from_logits(logits, T, E, k, ids, w, dev_status=None, stream=None):
    _check(lib().moe_topk_from_logits(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(dev_status), _stream(stream)),
           "moe_topk_from_logits")


# ----------------------------------------------------------------- permute

def moe_permute_workspace_size(T, k, E):
    return _size(lib().moe_permute_workspace_size, T, k, E)


def moe_permute(ids, T, k, E, offsets, perm, inv_perm, ws=None, ws_bytes=0, dev_status=None, stream=None):
    _check(lib().moe_permute(_ptr(ids), T, k, E, _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(ws), ws_bytes,
                             _ptr(dev_status), _stream(stream)), "moe_permute")


def moe_shard_ids(ids, n, e0, e_count, local_ids, stream=None):
    """ids of the shard holding experts [e0, e0 + e_count): local id, or MOE_ID_NOT_LOCAL for other shards."""
    _check(lib().moe_shard_ids(_ptr(ids), n, e0, e_count, _ptr(local_ids), _stream(stream)), "moe_shard_ids")


def moe_permute_noalloc(ids, T, k, E, offsets, perm, inv_perm, dev_status=None, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate (see the header)."""
    _check(lib().moe_permute_noalloc(_ptr(ids), T, k, E, _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(dev_status),
                                     _stream(stream)), "moe_permute_noalloc")


# ----------------------------------------------------------------- experts

def make_arena(bits, H, I, E, gu_codes, gu_scales, d_codes, d_scales) -> moe_expert_arena:
    return moe_expert_arena(bits, H, I, E, _ptr(gu_codes), _ptr(gu_scales), _ptr(d_codes), _ptr(d_scales))


def moe_expert_forward_workspace_size(arena: moe_expert_arena, T, k, path=MOE_PATH_AUTO):
    return _size(lib().moe_expert_forward_workspace_size, ctypes.byref(arena), T, k, path)


def moe_expert_forward(arena: moe_expert_arena, x_bf16, T, ids, w, k, offsets, perm, inv_perm, out, out_dtype=MOE_F32,
                       accumulate=False, path=MOE_PATH_AUTO, ws=None, ws_bytes=0, dev_status=None, stream=None):
    _check(lib().moe_expert_forward(ctypes.byref(arena), _ptr(x_bf16), T, _ptr(ids), _ptr(w), k, _ptr(offsets),
                                    _ptr(perm), _ptr(inv_perm), _ptr(out), out_dtype, int(accumulate), path, _ptr(ws),
                                    ws_bytes, _ptr(dev_status), _stream(stream)), "moe_expert_forward")


def moe_shared_expert_workspace_size(H, I, T):
    return _size(lib().moe_shared_expert_workspace_size, H, I, T)


def moe_shared_expert(wg, wu, wd, H, I, x_bf16, T, out, out_dtype=MOE_F32, accumulate=False, ws=None, ws_bytes=0,
                      dev_status=None, stream=None):
    _check(lib().moe_shared_expert(_ptr(wg), _ptr(wu), _ptr(wd), H, I, _ptr(x_bf16), T, _ptr(out), out_dtype,
                                   int(accumulate), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)),
           "moe_shared_expert")


def moe_f32_to_bf16(in_f32, out_bf16, n, stream=None):
    _check(lib().moe_f32_to_bf16(_ptr(in_f32), _ptr(out_bf16), n, _stream(stream)), "moe_f32_to_bf16")


def moe_decode_workspace_size(T, H, I, E, k, shared_I):
    return _size(lib().moe_decode_workspace_size, T, H, I, E, k, shared_I)


def moe_decode_forward(layers, x, T, k, rms_eps=RMS_EPS, ids_out=None, w_out=None, ws=None, ws_bytes=0,
                       dev_status=None, stream=None):
    """layers: a sequence of moe_layer_weights (host); x: [T][H] fp32 device tensor, updated in place."""
    arr = (moe_layer_weights * len(layers))(*layers)
    _check(lib().moe_decode_forward(arr, len(layers), _ptr(x), T, k, rms_eps, _ptr(ids_out), _ptr(w_out), _ptr(ws),
                                    ws_bytes, _ptr(dev_status), _stream(stream)), "moe_decode_forward")


def moe_decode_forward_ex(layers, x, T, k, rms_eps=RMS_EPS, route_tail_skip=0, hot_experts=None, ids_out=None,
                          w_out=None, ws=None, ws_bytes=0, dev_status=None, stream=None):
    """moe_decode_forward with options: route_tail_skip (rank threshold, 0 = off) and hot_experts (a device
    uint32 tensor [n_layers][(E + 31) // 32] of bit masks, or None)."""
    arr = (moe_layer_weights * len(layers))(*layers)
    opts = moe_decode_options(int(route_tail_skip), _ptr(hot_experts))
    _check(lib().moe_decode_forward_ex(arr, len(layers), _ptr(x), T, k, rms_eps, ctypes.byref(opts), _ptr(ids_out),
                                       _ptr(w_out), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)),
           "moe_decode_forward_ex")


def moe_rms_norm_bf16(x, out, T, H, eps=None, stream=None):
    _check(lib().moe_rms_norm_bf16(_ptr(x), _ptr(out), T, H, RMS_EPS if eps is None else eps, _stream(stream)),
           "moe_rms_norm_bf16")


def moe_selftest_barrier(extra_arrivals, timeout_ms, ws, ws_bytes, dev_status=None, stream=None):
    _check(lib().moe_selftest_barrier(extra_arrivals, timeout_ms, _ptr(ws), ws_bytes, _ptr(dev_status),
                                      _stream(stream)), "moe_selftest_barrier")


def header_functions():
    """Names of the functions include/moe_gb300.h declares."""
    import re

    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))
