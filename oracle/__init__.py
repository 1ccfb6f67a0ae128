"""The oracle: a plain, slow, scalar CPU statement of the routed-expert MoE layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library never calls it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (fp64, scalar, one loop per
definition); this module compiles it with gcc and exposes it through ctypes
on numpy arrays.  Routing decisions (top-k) are taken on fp32 logits, the
precision the GPU decides in.

Parity pins (tests/test_oracle_pins.py) cover every function here; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_INVALID_ARG = 1
ERR_NONFINITE = 6
ERR_BOUNDS = 7


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so (no fused multiply-add, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    L.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_fp16_to_double.restype = dbl
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = dbl
    L.oracle_dequant.argtypes = [i32, i32, ctypes.c_uint16]
    L.oracle_dequant.restype = dbl
    L.oracle_packed_row_bytes.argtypes = [i32, i64]
    L.oracle_packed_row_bytes.restype = i64
    L.oracle_pack.argtypes = [i32, i64, i64, P, P]
    L.oracle_pack.restype = i32
    L.oracle_unpack.argtypes = [i32, i64, i64, P, P]
    L.oracle_unpack.restype = i32
    L.oracle_router_logits.argtypes = [i32, i32, i32, P, P, P, P]
    L.oracle_router_logits.restype = None
    L.oracle_topk.argtypes = [i32, i32, i32, P, P, P]
    L.oracle_topk.restype = i32
    L.oracle_permute.argtypes = [i32, i32, i32, P, P, P, P]
    L.oracle_permute.restype = i32
    L.oracle_expert_ffn.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P]
    L.oracle_expert_ffn.restype = None
    L.oracle_shared_expert.argtypes = [i32, i32, P, P, P, P, P]
    L.oracle_shared_expert.restype = None
    L.oracle_moe_layer.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                                   i32, P, P, P, P]
    L.oracle_moe_layer.restype = i32
    L.oracle_rms_norm.argtypes = [i32, i32, P, dbl, P]
    L.oracle_rms_norm.restype = None
    L.oracle_fp16_round.argtypes = [dbl]
    L.oracle_fp16_round.restype = dbl
    L.oracle_e4m3_round.argtypes = [dbl]
    L.oracle_e4m3_round.restype = dbl
    L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_double.restype = dbl
    L.oracle_fp16_round_array.argtypes = [i64, P, P]
    L.oracle_fp16_round_array.restype = None
    L.oracle_e4m3_round_array.argtypes = [i64, P, P]
    L.oracle_e4m3_round_array.restype = None
    L.oracle_fp8_exponent.argtypes = [dbl]
    L.oracle_fp8_exponent.restype = i32
    L.oracle_expert_ffn_fp8.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P]
    L.oracle_expert_ffn_fp8.restype = i32
    L.oracle_moe_layer_fp8.argtypes = L.oracle_moe_layer.argtypes
    L.oracle_moe_layer_fp8.restype = i32
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def use_library(path):
    """Point this module at another build of the oracle source (returns the previous one).

    Used by the mutation tests, which compile deliberately broken copies of
    moe_oracle.c to check that the pins catch them.
    """
    global _lib
    with _lock:
        prev = _lib
        _lib = _bind(path) if isinstance(path, str) else path
    return prev


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: oracle status {status}")
        self.status = status


def fp16_to_double(bits: int) -> float:
    return lib().oracle_fp16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def dequant(bits: int, code: int, scale_fp16_bits: int) -> float:
    return lib().oracle_dequant(int(bits), int(code), int(scale_fp16_bits))


def packed_row_bytes(bits: int, cols: int) -> int:
    return int(lib().oracle_packed_row_bytes(bits, cols))


def pack(bits: int, codes: np.ndarray) -> np.ndarray:
    """codes uint8 [..., rows, cols] -> packed uint8 [..., rows, row_bytes]."""
    codes = _c(codes, np.uint8)
    cols = codes.shape[-1]
    rows = int(np.prod(codes.shape[:-1]))
    rb = packed_row_bytes(bits, cols)
    out = np.zeros(codes.shape[:-1] + (rb,), np.uint8)
    st = lib().oracle_pack(bits, rows, cols, _p(codes), _p(out))
    if st != OK:
        raise OracleError(st, "pack")
    return out


def unpack(bits: int, packed: np.ndarray, cols: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    rows = int(np.prod(packed.shape[:-1]))
    out = np.zeros(packed.shape[:-1] + (cols,), np.uint8)
    st = lib().oracle_unpack(bits, rows, cols, _p(packed), _p(out))
    if st != OK:
        raise OracleError(st, "unpack")
    return out


def router_logits(x_bf16: np.ndarray, w: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """x bf16 bits uint16 [T][H], w fp32 [E][H], bias fp32 [E] -> fp64 logits [T][E]."""
    x_bf16 = _c(x_bf16, np.uint16)
    w = _c(w, np.float32)
    T, H = x_bf16.shape
    E = w.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.zeros((T, E), np.float64)
    lib().oracle_router_logits(T, H, E, _p(x_bf16), _p(w), _p(b), _p(out))
    return out


def topk(logits_f32: np.ndarray, k: int):
    """fp32 logits [T][E] -> (ids int32 [T][k], w fp64 [T][k]); raises on NaN."""
    l32 = _c(logits_f32, np.float32)
    T, E = l32.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    st = lib().oracle_topk(T, E, k, _p(l32), _p(ids), _p(w))
    if st != OK:
        raise OracleError(st, "topk")
    return ids, w


def permute(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    st = lib().oracle_permute(T, k, E, _p(ids), _p(offsets), _p(perm), _p(inv))
    if st != OK:
        raise OracleError(st, "permute")
    return offsets, perm, inv


def expert_ffn(bits, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, x):
    """One routed expert on one token; x fp64 [H] -> y fp64 [H]."""
    gc, uc, dc = (_c(a, np.uint8) for a in (gate_codes, up_codes, down_codes))
    gs, us, ds = (_c(a, np.uint16) for a in (gate_scales, up_scales, down_scales))
    I, H = gc.shape
    x = _c(x, np.float64)
    y = np.zeros(H, np.float64)
    lib().oracle_expert_ffn(bits, H, I, _p(gc), _p(gs), _p(uc), _p(us), _p(dc), _p(ds), _p(x), _p(y))
    return y


def expert_ffn_fp8(bits, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, x):
    """The FP8 variant of one routed expert on one token (e4m3 operands with
    power-of-two scales, see oracle_expert_ffn_fp8); x fp64 [H] -> y fp64 [H]."""
    gc, uc, dc = (_c(a, np.uint8) for a in (gate_codes, up_codes, down_codes))
    gs, us, ds = (_c(a, np.uint16) for a in (gate_scales, up_scales, down_scales))
    I, H = gc.shape
    x = _c(x, np.float64)
    y = np.zeros(H, np.float64)
    st = lib().oracle_expert_ffn_fp8(bits, H, I, _p(gc), _p(gs), _p(uc), _p(us), _p(dc), _p(ds), _p(x), _p(y))
    if st != OK:
        raise OracleError(st, "expert_ffn_fp8")
    return y


def fp16_round(v) -> np.ndarray:
    """Nearest binary16 values (ties to even, past 65504 -> inf), as fp64."""
    v = _c(np.atleast_1d(v), np.float64)
    out = np.zeros_like(v)
    lib().oracle_fp16_round_array(v.size, _p(v), _p(out))
    return out


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 values (ties to even, saturating at +-448), as fp64."""
    v = _c(np.atleast_1d(v), np.float64)
    out = np.zeros_like(v)
    lib().oracle_e4m3_round_array(v.size, _p(v), _p(out))
    return out


def e4m3_to_double(b: int) -> float:
    return lib().oracle_e4m3_to_double(int(b))


def fp8_exponent(amax: float) -> int:
    return int(lib().oracle_fp8_exponent(float(amax)))


def shared_expert(wg, wu, wd, x):
    wg, wu, wd = (_c(a, np.uint16) for a in (wg, wu, wd))
    I, H = wg.shape
    x = _c(x, np.float64)
    y = np.zeros(H, np.float64)
    lib().oracle_shared_expert(H, I, _p(wg), _p(wu), _p(wd), _p(x), _p(y))
    return y


def moe_layer(bits, x_bf16, ids, w, gate_codes, gate_scales, up_codes, up_scales, down_codes,
              down_scales, shared=None, fp8=False):
    """Layer output fp64 [T][H] for given routing.  Arena arrays are [E][...] logical codes.
    fp8=True runs the routed experts in their FP8 variant (oracle_expert_ffn_fp8)."""
    x_bf16 = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    gc, uc, dc = (_c(a, np.uint8) for a in (gate_codes, up_codes, down_codes))
    gs, us, ds = (_c(a, np.uint16) for a in (gate_scales, up_scales, down_scales))
    T, H = x_bf16.shape
    k = ids.shape[1]
    E, I, _ = gc.shape
    if shared is None:
        Is, swg, swu, swd = 0, None, None, None
    else:
        swg, swu, swd = (_c(a, np.uint16) for a in shared)
        Is = swg.shape[0]
    out = np.zeros((T, H), np.float64)
    fn = lib().oracle_moe_layer_fp8 if fp8 else lib().oracle_moe_layer
    st = fn(bits, T, H, I, E, k, _p(x_bf16), _p(ids), _p(w), _p(gc), _p(gs),
            _p(uc), _p(us), _p(dc), _p(ds), Is, _p(swg), _p(swu), _p(swd), _p(out))
    if st != OK:
        raise OracleError(st, "moe_layer")
    return out


def rms_norm(x_f32: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) per row, fp64 result."""
    x = _c(x_f32, np.float32)
    T, H = x.shape
    y = np.zeros((T, H), np.float64)
    lib().oracle_rms_norm(T, H, _p(x), float(eps), _p(y))
    return y


def route_tail_skip(ids: np.ndarray, rank: int, hot=None) -> np.ndarray:
    """Pairs a verify window leaves out under the route-tail skip.

    "How Strata runs a 125-billion-parameter model on a single 12 GB to 24 GB
    graphics card", Step 2, "Verify-window route tail skip": an expert that
    every token of the window ranks at the very tail of its top-10 (ranks
    7, 8, 9 for the threshold 7) contributes almost nothing and is skipped;
    an expert ranked below the threshold by at least one token, or resident
    in the fast tier (`hot`), is kept.  Reading taken: a pair (t, j) is left
    out when j >= rank, its expert is not hot, and no pair of the window keeps
    that expert at a rank below the threshold; the kept pairs keep their
    weights.  rank 0 leaves nothing out.

    ids [T][k] int -> bool [T][k], True for a pair left out.
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    hot = set() if hot is None else set(int(e) for e in hot)
    out = np.zeros((T, k), bool)
    if rank <= 0:
        return out
    early = set()
    for t in range(T):
        for j in range(min(rank, k)):
            early.add(int(ids[t, j]))
    for t in range(T):
        for j in range(rank, k):
            e = int(ids[t, j])
            out[t, j] = e not in early and e not in hot
    return out
