"""ctypes binding of libkvq.so (include/kvq.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  The functions named like the C entry points take device pointers
(ints) or torch tensors (their data_ptr is passed); the lower-case helpers
below them allocate outputs with torch and call the same entry points.

If the library is missing or fails to load, importing this module raises:
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

from . import builder as _build

# ---- enums (include/kvq.h) ---------------------------------------------------
OK, EINVAL, ECUDA, EUNSUPPORTED, EWORKSPACE = 0, 1, 2, 3, 4
F32, BF16, I8, NONE = 0, 1, 2, 3
SYM, ASYM = 0, 1
ALONG_T, ALONG_C = 0, 1


class kvq_shape(ctypes.Structure):
    _fields_ = [("outer", ctypes.c_int64), ("T", ctypes.c_int64), ("C", ctypes.c_int64)]


class kvq_qparams(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("mode", ctypes.c_int32), ("qmin", ctypes.c_int32),
                ("qmax", ctypes.c_int32), ("axis", ctypes.c_int32), ("group", ctypes.c_int64),
                ("residual", ctypes.c_int64), ("scale_dtype", ctypes.c_int32),
                ("zero_dtype", ctypes.c_int32)]


class kvq_err(ctypes.Structure):
    _fields_ = [("rmse", ctypes.c_double), ("max_abs", ctypes.c_double), ("mean_abs", ctypes.c_double)]


class KvqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"kvq status {status}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libkvq.so is not built ({path}); run kv_cache_quantization_kvq_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    S, P = ctypes.POINTER(kvq_shape), ctypes.POINTER(kvq_qparams)
    psz = ctypes.POINTER(ctypes.c_size_t)
    i32 = ctypes.c_int
    sig = {
        "kvq_quantized_sizes": [S, i32, P, psz, psz, psz, psz, psz],
        "kvq_quantize": [vp, i32, S, P, vp, vp, vp, vp, vp, sz, vp],
        "kvq_dequantize": [vp, vp, vp, vp, S, P, vp, i32, vp],
        "kvq_error_stats": [vp, i32, vp, vp, vp, vp, S, P, vp, vp, sz, vp],
        "kvq_token_compression_ratio": [i64, i64, ctypes.POINTER(ctypes.c_double)],
        "kv_select_workspace": [i64, i64, psz],
        "kv_h2o_select": [vp, i64, i64, i64, i64, i64, vp, vp, vp, sz, vp],
        "kv_snapkv_select": [vp, i64, i64, i64, i64, i64, i64, vp, vp, vp, sz, vp],
        "kv_compact": [vp, i32, i64, i64, i64, vp, i64, vp, vp],
        "kv_compact_kv": [vp, vp, i32, i64, i64, i64, vp, i64, vp, vp, vp],
        "kvq_error_stats_noalloc": [vp, i32, vp, vp, vp, vp, S, P, vp, vp],
        "kvq_attend_workspace": [S, i64, psz],
        "kvq_attend_decode": [vp, i64, vp, vp, vp, vp, P, vp, vp, vp, vp, P, S, vp, vp, sz, vp],
        "kvq_rotate": [vp, i32, S, vp, i32, vp, i32, vp],
        "kvq_rotate_quantize": [vp, i32, S, vp, P, vp, vp, vp, vp, vp],
        "kvq_dequantize_rotate": [vp, vp, vp, vp, S, P, vp, vp, i32, vp],
        "kvq_append_workspace": [S, i32, P, i64, psz],
        "kvq_mixed_sizes": [S, psz, psz, psz],
        "kvq_mixed_quantize": [vp, vp, S, vp, vp, vp, vp],
        "kvq_mixed_dequantize": [vp, vp, vp, S, vp, vp],
        "kvq_wait_timeouts": [ctypes.POINTER(ctypes.c_uint64)],
        "kvq_append": [vp, i64, i32, S, P, i64, vp, vp, vp, vp, ctypes.POINTER(i64), ctypes.POINTER(i64), vp, sz,
                       vp],
        "kvq_append_kv_workspace": [S, i32, P, P, i64, psz],
        "kvq_append_kv": [vp, vp, i64, i32, S, P, P, i64, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(i64),
                          ctypes.POINTER(i64), vp, sz, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.kvq_compression_ratio.argtypes = [sz] * 5
    lib.kvq_compression_ratio.restype = ctypes.c_double
    lib.kvq_last_error.restype = ctypes.c_char_p
    lib.kvq_version.restype = ctypes.c_char_p
    return lib


LIB = _load()

# every symbol include/kvq.h declares
EXPORTS = ("kvq_quantized_sizes", "kvq_quantize", "kvq_dequantize", "kvq_error_stats",
           "kvq_compression_ratio", "kvq_token_compression_ratio", "kv_select_workspace",
           "kv_h2o_select", "kv_snapkv_select", "kv_compact", "kv_compact_kv", "kvq_last_error", "kvq_version",
           "kvq_error_stats_noalloc", "kvq_attend_workspace", "kvq_attend_decode", "kvq_rotate",
           "kvq_rotate_quantize", "kvq_dequantize_rotate", "kvq_append_kv_workspace", "kvq_append_kv",
           "kvq_append_workspace", "kvq_append", "kvq_mixed_sizes", "kvq_mixed_quantize", "kvq_mixed_dequantize",
           "kvq_wait_timeouts")

# size of the library's fixed scratch array behind kvq_error_stats_noalloc
NOALLOC_SCRATCH_BYTES = 1 << 20


def _check(status: int):
    if status != OK:
        raise KvqError(status, LIB.kvq_last_error().decode(errors="replace"))


def _ptr(p) -> Optional[int]:
    if p is None:
        return None
    if hasattr(p, "data_ptr"):
        return p.data_ptr() if p.numel() > 0 else None
    return int(p)


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


# ---- formats ----------------------------------------------------------------

@dataclass(frozen=True)
class QParams:
    """Quantized format (mirrors kvq_qparams)."""
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

    def c(self) -> kvq_qparams:
        return kvq_qparams(self.bits, self.mode, self.qmin, self.qmax, self.axis, self.group,
                           self.residual, self.scale_dtype, self.zero_dtype)


def _shape(shape) -> kvq_shape:
    outer, T, C = (int(v) for v in shape)
    return kvq_shape(outer, T, C)


# ---- the C entry points -------------------------------------------------------

def kvq_version() -> str:
    return LIB.kvq_version().decode()


def kvq_wait_timeouts() -> int:
    """Bounded waits of the library's kernels that gave up since it was loaded
    (synchronises the device); 0 in every correct run."""
    n = ctypes.c_uint64()
    _check(LIB.kvq_wait_timeouts(ctypes.byref(n)))
    return int(n.value)


def kvq_quantized_sizes(shape, x_dtype: int, qp: QParams):
    """(codes_B, scale_B, zero_B, resid_B, workspace_B)."""
    out = [ctypes.c_size_t() for _ in range(5)]
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_quantized_sizes(ctypes.byref(s), x_dtype, ctypes.byref(p), *[ctypes.byref(o) for o in out]))
    return tuple(int(o.value) for o in out)


def kvq_quantize(x, x_dtype, shape, qp: QParams, codes, scale, zero, resid, workspace, workspace_B, stream=None):
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_quantize(_ptr(x), x_dtype, ctypes.byref(s), ctypes.byref(p), _ptr(codes), _ptr(scale),
                            _ptr(zero), _ptr(resid), _ptr(workspace), int(workspace_B), _stream(stream)))


def kvq_dequantize(codes, scale, zero, resid, shape, qp: QParams, out, out_dtype, stream=None):
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_dequantize(_ptr(codes), _ptr(scale), _ptr(zero), _ptr(resid), ctypes.byref(s),
                              ctypes.byref(p), _ptr(out), out_dtype, _stream(stream)))


def kvq_error_stats(x, x_dtype, codes, scale, zero, resid, shape, qp: QParams, out_dev, workspace,
                    workspace_B, stream=None):
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_error_stats(_ptr(x), x_dtype, _ptr(codes), _ptr(scale), _ptr(zero), _ptr(resid),
                               ctypes.byref(s), ctypes.byref(p), _ptr(out_dev), _ptr(workspace),
                               int(workspace_B), _stream(stream)))


def kvq_error_stats_noalloc(x, x_dtype, codes, scale, zero, resid, shape, qp: QParams, out_dev, stream=None):
    """kvq_error_stats for callers that cannot allocate: no workspace argument,
    the library's fixed scratch array is used instead (see include/kvq.h)."""
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_error_stats_noalloc(_ptr(x), x_dtype, _ptr(codes), _ptr(scale), _ptr(zero), _ptr(resid),
                                       ctypes.byref(s), ctypes.byref(p), _ptr(out_dev), _stream(stream)))


def kvq_compression_ratio(orig_B, codes_B, scale_B, zero_B, resid_B) -> float:
    return float(LIB.kvq_compression_ratio(orig_B, codes_B, scale_B, zero_B, resid_B))


def kvq_token_compression_ratio(total_tokens: int, kept_tokens: int) -> float:
    out = ctypes.c_double()
    _check(LIB.kvq_token_compression_ratio(total_tokens, kept_tokens, ctypes.byref(out)))
    return float(out.value)


def kv_select_workspace(heads: int, T: int) -> int:
    out = ctypes.c_size_t()
    _check(LIB.kv_select_workspace(heads, T, ctypes.byref(out)))
    return int(out.value)


def kv_h2o_select(hist, heads, steps, T, budget, window, keep, scores, workspace, workspace_B, stream=None):
    _check(LIB.kv_h2o_select(_ptr(hist), heads, steps, T, budget, window, _ptr(keep), _ptr(scores),
                             _ptr(workspace), int(workspace_B), _stream(stream)))


def kv_snapkv_select(hist, heads, steps, T, obs_window, budget, window, keep, scores, workspace,
                     workspace_B, stream=None):
    _check(LIB.kv_snapkv_select(_ptr(hist), heads, steps, T, obs_window, budget, window, _ptr(keep),
                                _ptr(scores), _ptr(workspace), int(workspace_B), _stream(stream)))


def kv_compact(kv, dtype, heads, T, D, keep, K, out, stream=None):
    _check(LIB.kv_compact(_ptr(kv), dtype, heads, T, D, _ptr(keep), K, _ptr(out), _stream(stream)))


def kv_compact_kv(k, v, dtype, heads, T, D, keep, K, out_k, out_v, stream=None):
    _check(LIB.kv_compact_kv(_ptr(k), _ptr(v), dtype, heads, T, D, _ptr(keep), K, _ptr(out_k), _ptr(out_v),
                             _stream(stream)))


def kvq_attend_workspace(shape, group: int) -> int:
    s, n = _shape(shape), ctypes.c_size_t()
    _check(LIB.kvq_attend_workspace(ctypes.byref(s), int(group), ctypes.byref(n)))
    return n.value


def kvq_attend_decode(q, group, k_codes, k_scale, k_zero, k_resid, kqp: QParams, v_codes, v_scale, v_zero,
                      v_resid, vqp: QParams, shape, out, workspace, workspace_B, stream=None):
    s, pk, pv = _shape(shape), kqp.c(), vqp.c()
    _check(LIB.kvq_attend_decode(_ptr(q), int(group), _ptr(k_codes), _ptr(k_scale), _ptr(k_zero), _ptr(k_resid),
                                 ctypes.byref(pk), _ptr(v_codes), _ptr(v_scale), _ptr(v_zero), _ptr(v_resid),
                                 ctypes.byref(pv), ctypes.byref(s), _ptr(out), _ptr(workspace), int(workspace_B),
                                 _stream(stream)))


def kvq_rotate(x, x_dtype, shape, signs, inverse, out, out_dtype, stream=None):
    s = _shape(shape)
    _check(LIB.kvq_rotate(_ptr(x), x_dtype, ctypes.byref(s), _ptr(signs), int(bool(inverse)), _ptr(out), out_dtype,
                          _stream(stream)))


def kvq_rotate_quantize(x, x_dtype, shape, signs, qp: QParams, codes, scale, zero, resid, stream=None):
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_rotate_quantize(_ptr(x), x_dtype, ctypes.byref(s), _ptr(signs), ctypes.byref(p), _ptr(codes),
                                   _ptr(scale), _ptr(zero), _ptr(resid), _stream(stream)))


def kvq_dequantize_rotate(codes, scale, zero, resid, shape, qp: QParams, signs, out, out_dtype, stream=None):
    s, p = _shape(shape), qp.c()
    _check(LIB.kvq_dequantize_rotate(_ptr(codes), _ptr(scale), _ptr(zero), _ptr(resid), ctypes.byref(s),
                                     ctypes.byref(p), _ptr(signs), _ptr(out), out_dtype, _stream(stream)))


def kvq_append_workspace(shape, x_dtype, qp: QParams, block: int) -> int:
    s, p, n = _shape(shape), qp.c(), ctypes.c_size_t()
    _check(LIB.kvq_append_workspace(ctypes.byref(s), x_dtype, ctypes.byref(p), int(block), ctypes.byref(n)))
    return n.value


def kvq_append(x_new, n, x_dtype, shape, qp: QParams, block, codes, scale, zero, resid, tq, nres, workspace,
               workspace_B, stream=None):
    """Returns the updated (tq, nres) counters."""
    s, p = _shape(shape), qp.c()
    t, r = ctypes.c_int64(int(tq)), ctypes.c_int64(int(nres))
    _check(LIB.kvq_append(_ptr(x_new), int(n), x_dtype, ctypes.byref(s), ctypes.byref(p), int(block), _ptr(codes),
                          _ptr(scale), _ptr(zero), _ptr(resid), ctypes.byref(t), ctypes.byref(r), _ptr(workspace),
                          int(workspace_B), _stream(stream)))
    return t.value, r.value


def kvq_append_kv_workspace(shape, x_dtype, kqp: QParams, vqp: QParams, block: int) -> int:
    s, pk, pv, n = _shape(shape), kqp.c(), vqp.c(), ctypes.c_size_t()
    _check(LIB.kvq_append_kv_workspace(ctypes.byref(s), x_dtype, ctypes.byref(pk), ctypes.byref(pv), int(block),
                                       ctypes.byref(n)))
    return n.value


def kvq_append_kv(k_new, v_new, n, x_dtype, shape, kqp: QParams, vqp: QParams, block, k_bufs, v_bufs, tq, nres,
                  workspace, workspace_B, stream=None):
    """k_bufs / v_bufs: (codes, scale, zero, resid) of each cache.  Returns the
    updated (tq, nres) counters."""
    s, pk, pv = _shape(shape), kqp.c(), vqp.c()
    t, r = ctypes.c_int64(int(tq)), ctypes.c_int64(int(nres))
    _check(LIB.kvq_append_kv(_ptr(k_new), _ptr(v_new), int(n), x_dtype, ctypes.byref(s), ctypes.byref(pk),
                             ctypes.byref(pv), int(block), *[_ptr(x) for x in k_bufs], *[_ptr(x) for x in v_bufs],
                             ctypes.byref(t), ctypes.byref(r), _ptr(workspace), int(workspace_B), _stream(stream)))
    return t.value, r.value


class KVAppender:
    """Streaming append of one layer's K and V caches, one kvq_append_kv call
    per decode step.  The ctypes arguments that do not change between steps
    (shape, formats, buffers, workspace, stream) are built once; tq / nres are
    the shared counters."""

    def __init__(self, shape, x_dtype, kqp: QParams, vqp: QParams, block, k_bufs, v_bufs, workspace, tq=0, nres=0,
                 stream=None):
        self._s, self._pk, self._pv = _shape(shape), kqp.c(), vqp.c()
        self._t, self._r = ctypes.c_int64(int(tq)), ctypes.c_int64(int(nres))
        self._head = (x_dtype, ctypes.byref(self._s), ctypes.byref(self._pk), ctypes.byref(self._pv), int(block))
        self._tail = tuple(_ptr(x) for x in k_bufs) + tuple(_ptr(x) for x in v_bufs) + (
            ctypes.byref(self._t), ctypes.byref(self._r), _ptr(workspace), int(workspace.numel()), _stream(stream))
        self._fn = LIB.kvq_append_kv

    @property
    def tq(self) -> int:
        return self._t.value

    @property
    def nres(self) -> int:
        return self._r.value

    def set_counters(self, tq: int, nres: int):
        self._t.value, self._r.value = int(tq), int(nres)

    def append(self, k_new, v_new, n: int):
        """k_new, v_new: CUDA [outer, n, C] contiguous, the cache's dtype."""
        st = self._fn(k_new.data_ptr(), v_new.data_ptr(), n, *self._head, *self._tail)
        if st != OK:
            _check(st)


def kvq_mixed_sizes(shape):
    s = _shape(shape)
    a, b_, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(LIB.kvq_mixed_sizes(ctypes.byref(s), ctypes.byref(a), ctypes.byref(b_), ctypes.byref(c)))
    return a.value, b_.value, c.value


def kvq_mixed_quantize(x, tags, shape, stream_buf, off, tags2, stream=None):
    s = _shape(shape)
    _check(LIB.kvq_mixed_quantize(_ptr(x), _ptr(tags), ctypes.byref(s), _ptr(stream_buf), _ptr(off), _ptr(tags2),
                                  _stream(stream)))


def kvq_mixed_dequantize(stream_buf, off, tags2, shape, out, stream=None):
    s = _shape(shape)
    _check(LIB.kvq_mixed_dequantize(_ptr(stream_buf), _ptr(off), _ptr(tags2), ctypes.byref(s), _ptr(out),
                                    _stream(stream)))


def kvq_last_error() -> str:
    return LIB.kvq_last_error().decode(errors="replace")


# ---- allocating helpers (torch tensors on the current CUDA device) ------------

def torch_dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


@dataclass
class Quantized:
    """Buffers of one quantized tensor (device, caller-owned torch tensors)."""
    codes: "object"
    scale: "object"
    zero: "object"
    resid: "object"
    shape: tuple
    qp: QParams
    x_dtype: int


def _empty(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 0), dtype=torch.uint8, device=device)


def alloc_quantized(shape, x_dtype: int, qp: QParams, device="cuda"):
    cB, sB, zB, rB, wB = kvq_quantized_sizes(shape, x_dtype, qp)
    return (Quantized(_empty(cB, device), _empty(sB, device), _empty(zB, device), _empty(rB, device),
                      tuple(int(v) for v in shape), qp, x_dtype), _empty(wB, device))


def quantize(x, qp: QParams, out: Optional[Quantized] = None, workspace=None, stream=None) -> Quantized:
    """x: CUDA tensor [..., T, C] (leading dims flatten into outer), bf16 or fp32."""
    shape = (x.numel() // (x.shape[-1] * x.shape[-2]) if x.dim() >= 2 and x.shape[-1] * x.shape[-2] else 0,
             x.shape[-2], x.shape[-1])
    xd = torch_dtype_code(x)
    if out is None or workspace is None:
        out, workspace = alloc_quantized(shape, xd, qp, x.device)
    kvq_quantize(x, xd, shape, qp, out.codes, out.scale, out.zero, out.resid, workspace, workspace.numel(),
                 stream)
    return out


def dequantize(qt: Quantized, out=None, stream=None):
    import torch
    dt = torch.bfloat16 if qt.x_dtype == BF16 else torch.float32
    if out is None:
        out = torch.empty(qt.shape, dtype=dt, device=qt.codes.device)
    kvq_dequantize(qt.codes, qt.scale, qt.zero, qt.resid, qt.shape, qt.qp, out, qt.x_dtype, stream)
    return out


def error_stats(x, qt: Quantized, workspace=None, stream=None, out_dev=None):
    """Returns a device tensor of 3 doubles (rmse, max_abs, mean_abs)."""
    import torch
    if workspace is None:
        workspace = _empty(kvq_quantized_sizes(qt.shape, qt.x_dtype, qt.qp)[4], x.device)
    if out_dev is None:
        out_dev = torch.empty(3, dtype=torch.float64, device=x.device)
    kvq_error_stats(x, qt.x_dtype, qt.codes, qt.scale, qt.zero, qt.resid, qt.shape, qt.qp, out_dev,
                    workspace, workspace.numel(), stream)
    return out_dev


def h2o_select(hist, budget: int, window: int, workspace=None, scores=None, stream=None):
    """hist: CUDA float32 [heads, steps, T] -> (keep int32 [heads, min(B,T)], scores)."""
    import torch
    H, S, T = hist.shape
    keep = torch.empty((H, min(budget, T)), dtype=torch.int32, device=hist.device)
    if scores is None:
        scores = torch.empty((H, T), dtype=torch.float32, device=hist.device)
    if workspace is None:
        workspace = _empty(kv_select_workspace(H, T), hist.device)
    kv_h2o_select(hist, H, S, T, budget, window, keep, scores, workspace, workspace.numel(), stream)
    return keep, scores


def snapkv_select(hist, obs_window: int, budget: int, window: int, workspace=None, scores=None, stream=None):
    import torch
    H, S, T = hist.shape
    keep = torch.empty((H, min(budget, T)), dtype=torch.int32, device=hist.device)
    if scores is None:
        scores = torch.empty((H, T), dtype=torch.float32, device=hist.device)
    if workspace is None:
        workspace = _empty(kv_select_workspace(H, T), hist.device)
    kv_snapkv_select(hist, H, S, T, obs_window, budget, window, keep, scores, workspace, workspace.numel(),
                     stream)
    return keep, scores


def compact_kv(k, v, keep, out_k=None, out_v=None, stream=None):
    """k, v: CUDA [heads, T, D] of one dtype; keep: int32 [heads, K] -> (k', v') [heads, K, D]."""
    import torch
    H, T, D = k.shape
    K = keep.shape[1]
    code = {torch.float32: F32, torch.bfloat16: BF16, torch.int8: I8, torch.uint8: I8}[k.dtype]
    if out_k is None:
        out_k = torch.empty((H, K, D), dtype=k.dtype, device=k.device)
    if out_v is None:
        out_v = torch.empty((H, K, D), dtype=v.dtype, device=v.device)
    kv_compact_kv(k, v, code, H, T, D, keep, K, out_k, out_v, stream)
    return out_k, out_v


def compact(kv, keep, out=None, stream=None):
    """kv: CUDA [heads, T, D]; keep: int32 [heads, K] -> [heads, K, D]."""
    import torch
    H, T, D = kv.shape
    K = keep.shape[1]
    code = {torch.float32: F32, torch.bfloat16: BF16, torch.int8: I8, torch.uint8: I8}[kv.dtype]
    if out is None:
        out = torch.empty((H, K, D), dtype=kv.dtype, device=kv.device)
    kv_compact(kv, code, H, T, D, keep, K, out, stream)
    return out


def attend_decode(q, qk: Quantized, qv: Quantized, out=None, workspace=None, stream=None):
    """q: CUDA float32 [outer, group, C]; qk / qv: the quantized key and value
    caches of one bf16 [outer, T, C] shape -> float32 [outer, group, C], the
    attention output over the cache with the dequantization fused in."""
    import torch
    outer, group, C = q.shape
    if out is None:
        out = torch.empty((outer, group, C), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _empty(kvq_attend_workspace(qk.shape, group), q.device)
    kvq_attend_decode(q, group, qk.codes, qk.scale, qk.zero, qk.resid, qk.qp, qv.codes, qv.scale, qv.zero,
                      qv.resid, qv.qp, qk.shape, out, workspace, workspace.numel(), stream)
    return out


def rotate_quantize(x, signs, qp: QParams, out: Optional[Quantized] = None, stream=None) -> Quantized:
    """x: CUDA bf16 [..., T, C] -> the quantized rotated tensor (groups along
    C); the residual window holds rotated rows."""
    shape = (x.numel() // (x.shape[-1] * x.shape[-2]) if x.shape[-1] * x.shape[-2] else 0, x.shape[-2], x.shape[-1])
    if out is None:
        out, _ = alloc_quantized(shape, BF16, qp, x.device)
    kvq_rotate_quantize(x, torch_dtype_code(x), shape, signs, qp, out.codes, out.scale, out.zero, out.resid, stream)
    return out


def dequantize_rotate(qt: Quantized, signs, out=None, stream=None):
    """The inverse of rotate_quantize: x_hat rotated back, bf16."""
    import torch
    if out is None:
        out = torch.empty(qt.shape, dtype=torch.bfloat16, device=qt.codes.device)
    kvq_dequantize_rotate(qt.codes, qt.scale, qt.zero, qt.resid, qt.shape, qt.qp, signs, out, BF16, stream)
    return out


def rotate(x, signs, inverse=False, out=None, out_dtype=None, stream=None):
    """x: CUDA [..., T, C] bf16 or float32; signs: CUDA int8 [C] (+1 / -1) ->
    the randomized Hadamard rotation of every row (or its inverse)."""
    import torch
    shape = (x.numel() // (x.shape[-1] * x.shape[-2]) if x.shape[-1] * x.shape[-2] else 0, x.shape[-2], x.shape[-1])
    od = torch_dtype_code(x) if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16 if od == BF16 else torch.float32, device=x.device)
    kvq_rotate(x, torch_dtype_code(x), shape, signs, inverse, out, od, stream)
    return out

