"""Shared helpers of the GPU parity tests: move host buffers to the device,
run the CUDA path through the C ABI, and bring results back as numpy."""
import numpy as np

import oracle as O


def kb():
    from kv_cache_quantization_kvq_gb300 import build
    build()
    from kv_cache_quantization_kvq_gb300 import binding
    return binding


def to_device(a: np.ndarray, x_dtype: int):
    """float32 -> torch float32; uint16 bf16 bits -> torch bfloat16 (same bits)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if x_dtype == O.BF16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def to_host(t, np_dtype=None) -> np.ndarray:
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    a = t.numpy()
    return a.view(np_dtype) if np_dtype is not None else a


def kq_of(b, oq: O.QParams):
    return b.QParams(oq.bits, oq.mode, oq.qmin, oq.qmax, oq.axis, oq.group, oq.residual,
                     oq.scale_dtype, oq.zero_dtype)


def meta_np_dtype(code):
    return {O.F32: np.float32, O.BF16: np.uint16, O.I8: np.int8}[code]
