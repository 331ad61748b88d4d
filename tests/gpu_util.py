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


# ---------------------------------------------------------------- write guards
#
# Every device buffer a call may write is carved out of a larger allocation
# whose bytes before and after the window hold a canary pattern.  A kernel
# that stores outside its output (a ragged last group, a partial channel
# block, a tail CTA) changes a canary byte, which check() reports; the exact
# window comparisons of the parity tests cannot see such stores.

CANARY_PAD = 256          # keeps every window 256-byte aligned (workspace alignment)


def canary_pattern(n: int) -> np.ndarray:
    """A position-dependent byte pattern (no run of equal bytes, never all 0)."""
    return ((np.arange(n, dtype=np.uint32) * 37 + 0xA5) & 0xFF).astype(np.uint8)


class Guarded:
    """Allocates guarded device windows and checks their canaries."""

    def __init__(self):
        self.items = []

    def alloc(self, nbytes: int, offset: int = 0, fill=None):
        """A uint8 window of nbytes at byte `offset` past a 256-byte aligned
        boundary, CANARY_PAD canary bytes (plus offset) before it and
        CANARY_PAD after it.  The window itself starts as canary bytes too
        (an output byte the call never writes then fails its comparison),
        unless fill (an int byte value) is given."""
        import torch
        if nbytes == 0:
            return None
        total = CANARY_PAD + offset + nbytes + CANARY_PAD
        pat = canary_pattern(total)
        raw = torch.from_numpy(pat.copy()).to("cuda")
        start = CANARY_PAD + offset
        win = raw[start:start + nbytes]
        if fill is not None:
            win.fill_(fill)
        self.items.append((raw, start, nbytes, pat))
        return win

    def check(self, what: str = ""):
        import torch
        torch.cuda.synchronize()
        for raw, start, n, pat in self.items:
            h = raw.cpu().numpy()
            before, after = h[:start], h[start + n:]
            bad_b = np.nonzero(before != pat[:start])[0]
            bad_a = np.nonzero(after != pat[start + n:])[0]
            assert bad_b.size == 0, f"{what}: store {start - bad_b[0]} bytes before a {n}-byte window"
            assert bad_a.size == 0, f"{what}: store {bad_a[0]} bytes past the end of a {n}-byte window"
