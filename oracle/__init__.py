"""CPU oracle for the KV-cache compression hot path -- TEST INFRASTRUCTURE ONLY.

This package wraps ``kvq_oracle.c`` (plain scalar C, float32 arithmetic with no
fused multiply-add, binary64 accumulation for the error statistics) with
ctypes and numpy.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it.  The CUDA library and its Python
binding never do: the two implementations share no code.

Sources (page title, section) are cited in ``kvq_oracle.c``; the functions
here only marshal numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libkvq_oracle.so")

# dtype / mode / axis codes of the oracle's own entry points
F32, BF16, I8, NONE = 0, 1, 2, 3
SYM, ASYM = 0, 1
ALONG_T, ALONG_C = 0, 1
OK, EINVAL = 0, 1

_ITEMSIZE = {F32: 4, BF16: 2, I8: 1, NONE: 0}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE binary32, no contraction, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fno-finite-math-only", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [("outer", ctypes.c_int64), ("T", ctypes.c_int64), ("C", ctypes.c_int64),
                ("bits", ctypes.c_int32), ("mode", ctypes.c_int32), ("qmin", ctypes.c_int32),
                ("qmax", ctypes.c_int32), ("axis", ctypes.c_int32),
                ("group", ctypes.c_int64), ("residual", ctypes.c_int64),
                ("scale_dtype", ctypes.c_int32), ("zero_dtype", ctypes.c_int32)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_Params)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        p64 = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_sizes.argtypes = [P, i32, p64, p64, p64, p64]
        lib.oracle_compression_ratio.argtypes = [i64] * 5
        lib.oracle_compression_ratio.restype = ctypes.c_double
        lib.oracle_token_compression_ratio.argtypes = [i64, i64, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_quantize.argtypes = [vp, i32, P, vp, vp, vp, vp]
        lib.oracle_dequantize.argtypes = [vp, vp, vp, vp, P, vp, i32]
        lib.oracle_error_stats.argtypes = [vp, i32, vp, vp, vp, vp, P, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_h2o_select.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp]
        lib.oracle_snapkv_select.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp, vp]
        lib.oracle_compact.argtypes = [vp, i64, i64, i64, i64, vp, i64, vp]
        lib.oracle_dequantize_f64.argtypes = [vp, vp, vp, vp, P, i32, vp]
        lib.oracle_attend.argtypes = [vp, i64, vp, vp, i64, i64, i64, vp]
        lib.oracle_rotate.argtypes = [vp, i64, i64, vp, i32, vp]
        lib.oracle_rotate_fwht32.argtypes = [vp, i32, i64, i64, vp, i32, vp, i32]
        for f in ("oracle_sizes", "oracle_token_compression_ratio", "oracle_quantize",
                  "oracle_dequantize", "oracle_error_stats", "oracle_h2o_select",
                  "oracle_snapkv_select", "oracle_compact", "oracle_dequantize_f64", "oracle_attend", "oracle_rotate",
                  "oracle_rotate_fwht32"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(ValueError):
    """The oracle rejected its arguments (the pages' ValueError cases)."""


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what}: invalid arguments (status {rc})")


@dataclass(frozen=True)
class QParams:
    """Quantization format: bit width, mode, integer range, grouping, residual."""
    bits: int
    mode: int = SYM
    qmin: int = 0
    qmax: int = 0
    axis: int = ALONG_T
    group: int = 0
    residual: int = 0
    scale_dtype: int = F32
    zero_dtype: int = NONE

    @staticmethod
    def sym(bits, axis=ALONG_T, group=0, residual=0, scale_dtype=F32, qmax=None):
        q = (1 << (bits - 1)) - 1 if qmax is None else qmax
        return QParams(bits, SYM, -q, q, axis, group, residual, scale_dtype, NONE)

    @staticmethod
    def asym(bits, qmin, qmax, axis=ALONG_T, group=0, residual=0, scale_dtype=F32, zero_dtype=I8):
        return QParams(bits, ASYM, qmin, qmax, axis, group, residual, scale_dtype, zero_dtype)

    def c(self, shape) -> _Params:
        outer, T, C = shape
        return _Params(outer, T, C, self.bits, self.mode, self.qmin, self.qmax, self.axis,
                       self.group, self.residual, self.scale_dtype, self.zero_dtype)


def np_dtype(code: int):
    return {F32: np.float32, BF16: np.uint16, I8: np.int8}[code]


def sizes(shape, x_dtype: int, qp: QParams):
    """(codes_B, scale_B, zero_B, resid_B) of the quantized representation."""
    out = [ctypes.c_int64() for _ in range(4)]
    p = qp.c(shape)
    _check(_load().oracle_sizes(ctypes.byref(p), x_dtype, *[ctypes.byref(o) for o in out]), "sizes")
    return tuple(int(o.value) for o in out)


def compression_ratio(orig_B, codes_B, scale_B, zero_B, resid_B) -> float:
    return float(_load().oracle_compression_ratio(orig_B, codes_B, scale_B, zero_B, resid_B))


def token_compression_ratio(total_tokens: int, kept_tokens: int) -> float:
    out = ctypes.c_double()
    _check(_load().oracle_token_compression_ratio(total_tokens, kept_tokens, ctypes.byref(out)),
           "token_compression_ratio")
    return float(out.value)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Quantized:
    codes: np.ndarray   # uint8, packed
    scale: np.ndarray   # float32 or uint16 (bf16 bits)
    zero: np.ndarray    # int8 / uint16 (bf16 bits) / float32 / empty
    resid: np.ndarray   # source dtype, [outer, R, C]


def quantize(x: np.ndarray, x_dtype: int, qp: QParams) -> Quantized:
    """x: [outer, T, C] as float32 (F32) or uint16 bf16 bits (BF16)."""
    x = np.ascontiguousarray(x)
    assert x.ndim == 3 and x.dtype == np_dtype(x_dtype)
    shape = x.shape
    cB, sB, zB, rB = sizes(shape, x_dtype, qp)
    codes = np.zeros(cB, np.uint8)
    scale = np.zeros(sB // _ITEMSIZE[qp.scale_dtype], np_dtype(qp.scale_dtype))
    zero = (np.zeros(zB // _ITEMSIZE[qp.zero_dtype], np_dtype(qp.zero_dtype))
            if qp.zero_dtype != NONE else np.zeros(0, np.uint8))
    resid = np.zeros(rB // _ITEMSIZE[x_dtype], np_dtype(x_dtype))
    p = qp.c(shape)
    _check(_load().oracle_quantize(_ptr(x), x_dtype, ctypes.byref(p), _ptr(codes), _ptr(scale),
                                   _ptr(zero), _ptr(resid)), "quantize")
    return Quantized(codes, scale, zero, resid)


def dequantize(qt: Quantized, shape, qp: QParams, out_dtype: int) -> np.ndarray:
    out = np.zeros(shape, np_dtype(out_dtype))
    p = qp.c(shape)
    _check(_load().oracle_dequantize(_ptr(qt.codes), _ptr(qt.scale), _ptr(qt.zero), _ptr(qt.resid),
                                     ctypes.byref(p), _ptr(out), out_dtype), "dequantize")
    return out


def error_stats(x: np.ndarray, x_dtype: int, qt: Quantized, qp: QParams):
    """(rmse, max_abs, mean_abs) in binary64."""
    x = np.ascontiguousarray(x)
    out = (ctypes.c_double * 3)()
    p = qp.c(x.shape)
    _check(_load().oracle_error_stats(_ptr(x), x_dtype, _ptr(qt.codes), _ptr(qt.scale),
                                      _ptr(qt.zero), _ptr(qt.resid), ctypes.byref(p), out),
           "error_stats")
    return float(out[0]), float(out[1]), float(out[2])


def h2o_select(hist: np.ndarray, budget: int, window: int):
    """hist [heads, steps, T] float32 -> (keep [heads, min(B,T)] int32, scores [heads, T])."""
    hist = np.ascontiguousarray(hist, dtype=np.float32)
    H, S, T = hist.shape
    keep = np.zeros((H, min(budget, T)), np.int32)
    scores = np.zeros((H, T), np.float32)
    _check(_load().oracle_h2o_select(_ptr(hist), H, S, T, budget, window, _ptr(keep), _ptr(scores)),
           "h2o_select")
    return keep, scores


def snapkv_select(hist: np.ndarray, obs_window: int, budget: int, window: int):
    hist = np.ascontiguousarray(hist, dtype=np.float32)
    H, S, T = hist.shape
    keep = np.zeros((H, min(budget, T)), np.int32)
    scores = np.zeros((H, T), np.float32)
    _check(_load().oracle_snapkv_select(_ptr(hist), H, S, T, obs_window, budget, window,
                                        _ptr(keep), _ptr(scores)), "snapkv_select")
    return keep, scores


def compact(kv: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """kv [heads, T, D] (any itemsize), keep [heads, K] -> [heads, K, D]."""
    kv = np.ascontiguousarray(kv)
    keep = np.ascontiguousarray(keep, dtype=np.int32)
    H, T, D = kv.shape
    K = keep.shape[1]
    out = np.zeros((H, K, D), kv.dtype)
    _check(_load().oracle_compact(_ptr(kv), kv.itemsize, H, T, D, _ptr(keep), K, _ptr(out)), "compact")
    return out


def dequantize_f64(qt: Quantized, shape, qp: QParams, x_dtype: int) -> np.ndarray:
    """The cache rows in binary64: s * (q - zp) for quantized tokens, the
    residual rows (stored in x_dtype) widened."""
    out = np.zeros(shape, np.float64)
    p = qp.c(shape)
    _check(_load().oracle_dequantize_f64(_ptr(qt.codes), _ptr(qt.scale), _ptr(qt.zero), _ptr(qt.resid),
                                         ctypes.byref(p), x_dtype, _ptr(out)), "dequantize_f64")
    return out


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """q [outer, group, C], k / v [outer, T, C] (binary64) -> y [outer, group, C]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    outer, group, C = q.shape
    T = k.shape[1]
    assert k.shape == (outer, T, C) and v.shape == (outer, T, C)
    out = np.zeros((outer, group, C), np.float64)
    _check(_load().oracle_attend(_ptr(q), group, _ptr(k), _ptr(v), outer, T, C, _ptr(out)), "attend")
    return out


def rotate(x: np.ndarray, signs: np.ndarray, inverse: bool = False) -> np.ndarray:
    """Randomized Hadamard rotation of the last axis (binary64): forward
    (1/sqrt(C)) H (signs * x), inverse signs * ((1/sqrt(C)) H y)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    C = x.shape[-1]
    signs = np.ascontiguousarray(signs, dtype=np.int8)
    assert signs.shape == (C,)
    out = np.zeros_like(x)
    _check(_load().oracle_rotate(_ptr(x), x.size // C if C else 0, C, _ptr(signs), int(inverse), _ptr(out)),
           "rotate")
    return out


def rotate_fwht32(x: np.ndarray, x_dtype: int, signs: np.ndarray, inverse: bool = False,
                  out_dtype: int = F32) -> np.ndarray:
    """The rotation as the binary32 fast Walsh-Hadamard transform (stages of
    channel bit 1, 2, 4, ... in that order, then the multiply by the binary32
    nearest 1/sqrt(C)).  x: float32 values (F32) or bf16 bit patterns (BF16,
    uint16); returns float32 values or bf16 bit patterns (out_dtype)."""
    x = np.ascontiguousarray(x, dtype=np.uint16 if x_dtype == BF16 else np.float32)
    C = x.shape[-1]
    signs = np.ascontiguousarray(signs, dtype=np.int8)
    assert signs.shape == (C,)
    out = np.zeros(x.shape, np.uint16 if out_dtype == BF16 else np.float32)
    _check(_load().oracle_rotate_fwht32(_ptr(x), x_dtype, x.size // C if C else 0, C, _ptr(signs), int(inverse),
                                        _ptr(out), out_dtype), "rotate_fwht32")
    return out


# ---- bf16 helpers for tests (bit patterns held in uint16) -----------------

def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)
