"""GB300 (sm_103a) KV-cache compression hot path.

Quantize / dequantize (symmetric and asymmetric INT8/INT4/INT2, per-channel
and per-group scales, KIVI axes, bf16 residual window, bit packing), error
and compression-ratio metrics, H2O / SnapKV keep-set selection and the
compaction gather -- all in hand-written CUDA kernels behind the C ABI of
include/kvq.h.  ``binding`` is the ctypes layer over that library; it refuses
to import when the library is not built (there is no CPU fallback).
"""
from .builder import build  # noqa: F401

__all__ = ["build"]
