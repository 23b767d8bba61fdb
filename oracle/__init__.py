"""CPU oracle for NVFP4 block quantization (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does, and this
package never imports the product library.

The arithmetic lives in ``nvfp4_oracle.cpp`` (plain C++, IEEE fp32, no FMA
contraction, no flush-to-zero); this module only compiles it with g++ and
marshals numpy arrays through ctypes.  Arrays are numpy: fp32 inputs as
``float32``, bf16 inputs as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.cpp")
_HDR = os.path.join(_HERE, "nvfp4_oracle.h")
_LIB = os.path.join(_HERE, "liboracle_nvfp4.so")
# a prebuilt oracle library to load instead (the mutation test uses this to
# load copies of the oracle with planted mistakes)
_LIB_OVERRIDE = os.environ.get("NVFP4_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
BLOCK_1X16, BLOCK_16X16 = 0, 1
RTN, SR, RTN_STD = 0, 1, 2
GAMAX_NONE, GAMAX_TENSOR, GAMAX_ROW, GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN = 0, 1, 2, 3, 4
ERR_NONE, ERR_MAE, ERR_MSE = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle_nvfp4.so`` next to its source."""
    with _lock:
        stale = (not os.path.exists(_LIB) or
                 os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                   "-fno-finite-math-only", "-Wall", "-pthread", "-shared", "-fPIC", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if _LIB_OVERRIDE:
        lib = ctypes.CDLL(_LIB_OVERRIDE)
    else:
        build()
        lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i64, u64, i32, f32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_float
    lib.orc_e4m3_decode.restype = f32
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [f32]
    lib.orc_e2m1_value.restype = f32
    lib.orc_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_encode_rn.restype = ctypes.c_uint8
    lib.orc_e2m1_encode_rn.argtypes = [f32]
    lib.orc_e2m1_encode_sr.restype = ctypes.c_uint8
    lib.orc_e2m1_encode_sr.argtypes = [f32, ctypes.c_double]
    lib.orc_bf16_to_f32.restype = f32
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_philox4x32_10.restype = None
    lib.orc_philox4x32_10.argtypes = [P, P, P]
    lib.orc_sr_uniform.restype = ctypes.c_double
    lib.orc_sr_uniform.argtypes = [u64, u64, u64]
    lib.orc_global_scales.restype = None
    lib.orc_global_scales.argtypes = [f32, f32, P, P]
    lib.orc_amax.restype = None
    lib.orc_amax.argtypes = [P, i64, i64, i32, P, i32, P]
    lib.orc_scales_to_mma.restype = None
    lib.orc_scales_to_mma.argtypes = [P, i64, i64, P]
    lib.orc_quantize.restype = i32
    lib.orc_quantize.argtypes = [P, i64, i64, i32, i32, i32, P, u64, u64, i64, i32, P, i32, f32,
                                 P, P, P, P]
    lib.orc_dequantize.restype = i32
    lib.orc_dequantize.argtypes = [P, P, i64, i64, i32, P, f32, P, i32]
    lib.orc_qdq.restype = i32
    lib.orc_qdq.argtypes = [P, i64, i64, i32, i32, i32, P, u64, u64, i64, i32, P, i32, f32, P, P, P]
    for name in ("orc_e4m3_encode_n", "orc_e2m1_encode_rn_n", "orc_f32_to_bf16_n"):
        getattr(lib, name).restype = None
        getattr(lib, name).argtypes = [P, i64, P]
    lib.orc_e2m1_encode_sr_n.restype = None
    lib.orc_e2m1_encode_sr_n.argtypes = [P, P, i64, P]
    lib.orc_sr_uniform_n.restype = None
    lib.orc_sr_uniform_n.argtypes = [u64, u64, P, i64, P]
    lib.orc_e2m1_encode_rn_bits.restype = None
    lib.orc_e2m1_encode_rn_bits.argtypes = [ctypes.c_uint32, i64, P]
    lib.orc_set_threads.restype = i32
    lib.orc_set_threads.argtypes = [i32]
    lib.orc_get_threads.restype = i32
    lib.orc_get_threads.argtypes = []
    lib.orc_fp_env_ok.restype = i32
    lib.orc_fp_env_ok.argtypes = []
    if not lib.orc_fp_env_ok():
        raise RuntimeError("oracle: subnormal fp32 arithmetic is flushed on this host")
    _lib = lib
    return lib


def set_threads(n: int) -> int:
    """Worker threads for the oracle's loops over independent rows, bands and
    elements (0: one per hardware thread); returns the previous count.  The
    results do not depend on it (each block's arithmetic is unchanged)."""
    return int(_load().orc_set_threads(int(n)))


def threads() -> int:
    return int(_load().orc_get_threads())


class using_threads:
    """``with oracle.using_threads(n): ...`` runs the oracle on n threads."""

    def __init__(self, n: int):
        self.n = n

    def __enter__(self):
        self.old = set_threads(self.n)
        return threads()

    def __exit__(self, *exc):
        set_threads(self.old)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_of(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle input must be float32 or uint16 (bf16 bits), got {x.dtype}")


# ---- scalar codecs (vectorised by looping in C) ---------------------------------------
def e4m3_decode(b) -> np.ndarray:
    lib = _load()
    b = np.asarray(b, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(v)) for v in b.ravel()], np.float32).reshape(b.shape)


def e4m3_encode(s) -> np.ndarray:
    lib = _load()
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty(s.shape, np.uint8)
    lib.orc_e4m3_encode_n(_ptr(s), s.size, _ptr(out))
    return out


def e2m1_value(code) -> np.ndarray:
    lib = _load()
    c = np.asarray(code, dtype=np.uint8)
    return np.array([lib.orc_e2m1_value(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def e2m1_encode_rn(v) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib.orc_e2m1_encode_rn_n(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_encode_sr(v, u) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    u = np.ascontiguousarray(np.broadcast_to(u, v.shape), dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    lib.orc_e2m1_encode_sr_n(_ptr(v), _ptr(u), v.size, _ptr(out))
    return out


def e2m1_encode_rn_bits(first: int, n: int) -> np.ndarray:
    """Codes of the n consecutive fp32 bit patterns starting at ``first``."""
    lib = _load()
    out = np.empty(n, np.uint8)
    lib.orc_e2m1_encode_rn_bits(first, n, _ptr(out))
    return out


def f32_to_bf16(f) -> np.ndarray:
    lib = _load()
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    lib.orc_f32_to_bf16_n(_ptr(f), f.size, _ptr(out))
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_uniform(seed: int, step: int, idx) -> np.ndarray:
    lib = _load()
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.shape, np.float64)
    lib.orc_sr_uniform_n(seed, step, _ptr(idx), idx.size, _ptr(out))
    return out


def global_scales(A: float, bound: float):
    lib = _load()
    e = ctypes.c_float()
    d = ctypes.c_float()
    lib.orc_global_scales(A, bound, ctypes.byref(e), ctypes.byref(d))
    return np.float32(e.value), np.float32(d.value)


def amax(x: np.ndarray, residual: np.ndarray | None = None, per_row: bool = False) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x)
    M, K = x.shape
    out = np.zeros(M if per_row else 1, np.float32)
    r = None if residual is None else np.ascontiguousarray(residual, dtype=np.float32)
    lib.orc_amax(_ptr(x), M, K, _dtype_of(x), _ptr(r), GAMAX_ROW if per_row else GAMAX_TENSOR,
                 _ptr(out))
    return out


# ---- the three calls ------------------------------------------------------------------
def _default_bound(err_mode: int, scale_bound):
    if scale_bound is not None:
        return float(scale_bound)
    return 448.0 if err_mode == ERR_NONE else 256.0


def quantize(x: np.ndarray, *, block: int = BLOCK_1X16, rounding: int = RTN,
             residual: np.ndarray | None = None, seed: int = 0, step: int = 0,
             row_offset: int = 0, gamax_mode: int = GAMAX_NONE, gamax=None,
             err_mode: int = ERR_NONE, scale_bound: float | None = None, colwise: bool = False):
    """Returns dict(codes, scales[, codes_col, scales_col], gamax).  ``residual``
    (float32, contiguous) is updated in place, as the library does.  The bound
    defaults to 448 for the plain quantizer and 256 for four-over-six (the
    four-over-six page's default)."""
    lib = _load()
    scale_bound = _default_bound(err_mode, scale_bound)
    x = np.ascontiguousarray(x)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    codes_col = np.zeros((K, M // 2), np.uint8) if colwise else None
    scales_col = np.zeros((K, M // 16), np.uint8) if colwise else None
    if gamax_mode in (GAMAX_TENSOR, GAMAX_ROW):
        g = np.zeros(1 if gamax_mode == GAMAX_TENSOR else max(M, 1), np.float32)
    elif gamax_mode in (GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN):
        g = np.ascontiguousarray(gamax, dtype=np.float32).reshape(-1).copy()
    else:
        g = None
    if residual is not None:
        assert residual.dtype == np.float32 and residual.flags["C_CONTIGUOUS"]
    rc = lib.orc_quantize(_ptr(x), M, K, _dtype_of(x), block, rounding, _ptr(residual),
                          seed, step, row_offset, gamax_mode, _ptr(g), err_mode, scale_bound,
                          _ptr(codes), _ptr(scales), _ptr(codes_col), _ptr(scales_col))
    if rc:
        raise ValueError("oracle: argument combination not defined by the method")
    out = {"codes": codes, "scales": scales, "gamax": g}
    if colwise:
        out["codes_col"] = codes_col
        out["scales_col"] = scales_col
    return out


def scales_to_mma(scales: np.ndarray) -> np.ndarray:
    """Row-major scale bytes [rows, cols] -> the matrix-multiply layout (flat bytes)."""
    lib = _load()
    s = np.ascontiguousarray(scales, np.uint8)
    rows, cols = s.shape
    out = np.zeros(((rows + 127) // 128 * 128) * ((cols + 3) // 4 * 4), np.uint8)
    lib.orc_scales_to_mma(_ptr(s), rows, cols, _ptr(out))
    return out


def mm_reference(codes_a: np.ndarray, scales_a: np.ndarray, codes_b: np.ndarray, scales_b: np.ndarray,
                 M: int, N: int, K: int, gamax_a=None, gamax_b=None, scale_bound: float = 448.0):
    """The plain definition of the FP4 product ("fp4-train", API: fp4_mm, a @ b^T,
    and Correctness: equal to the dequantize path): (deq(A) deq(B)^T) with each
    operand dequantized without its global scale, in float64, times both fp32
    decode scales.  Row-major scales [M, K/16], [N, K/16]; returns float64 [M, N]."""
    da = dequantize(codes_a, scales_a, M, K, out_dtype=F32).astype(np.float64)
    db = dequantize(codes_b, scales_b, N, K, out_dtype=F32).astype(np.float64)
    alpha = 1.0
    for g in (gamax_a, gamax_b):
        if g is not None:
            alpha *= float(global_scales(float(np.asarray(g).ravel()[0]), scale_bound)[1])
    return (da @ db.T) * alpha


def dequantize(codes: np.ndarray, scales: np.ndarray, M: int, K: int, *,
               gamax_mode: int = GAMAX_NONE, gamax=None, scale_bound: float = 448.0,
               out_dtype: int = BF16) -> np.ndarray:
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    g = None if gamax is None else np.ascontiguousarray(gamax, dtype=np.float32).reshape(-1)
    out = np.empty((M, K), np.uint16 if out_dtype == BF16 else np.float32)
    rc = lib.orc_dequantize(_ptr(codes), _ptr(scales), M, K, gamax_mode, _ptr(g), scale_bound,
                            _ptr(out), out_dtype)
    if rc:
        raise ValueError("oracle: bad dequantize arguments")
    return out


def qdq(x: np.ndarray, *, block: int = BLOCK_1X16, rounding: int = RTN,
        residual: np.ndarray | None = None, seed: int = 0, step: int = 0, row_offset: int = 0,
        gamax_mode: int = GAMAX_NONE, gamax=None, err_mode: int = ERR_NONE,
        scale_bound: float | None = None):
    """Returns dict(out (bf16 bits, uint16), codes, scales, gamax)."""
    lib = _load()
    scale_bound = _default_bound(err_mode, scale_bound)
    x = np.ascontiguousarray(x)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    out = np.empty((M, K), np.uint16)
    if gamax_mode in (GAMAX_TENSOR, GAMAX_ROW):
        g = np.zeros(1 if gamax_mode == GAMAX_TENSOR else max(M, 1), np.float32)
    elif gamax_mode in (GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN):
        g = np.ascontiguousarray(gamax, dtype=np.float32).reshape(-1).copy()
    else:
        g = None
    rc = lib.orc_qdq(_ptr(x), M, K, _dtype_of(x), block, rounding, _ptr(residual), seed, step,
                     row_offset, gamax_mode, _ptr(g), err_mode, scale_bound, _ptr(codes),
                     _ptr(scales), _ptr(out))
    if rc:
        raise ValueError("oracle: argument combination not defined by the method")
    return {"out": out, "codes": codes, "scales": scales, "gamax": g}
