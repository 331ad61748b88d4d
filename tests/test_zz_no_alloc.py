"""kvq_error_stats_noalloc: the error statistics for callers that cannot
allocate device memory (for example a serving loop whose pool owns all device
memory, or code that must not call cudaMalloc on its hot path because it can
synchronise the device).  It uses the library's fixed scratch array instead
of a workspace; its results must match kvq_error_stats given a workspace, on
two calls in a row (the array keeps the previous call's contents).

This file is collected after every other parity test (only the wait-timeout
check follows), so that a run stopping at the first failure has already run
them; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

RTOL = 1e-5


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_quantization_kvq_gb300 import build
    build()
    from kv_cache_quantization_kvq_gb300 import binding
    return binding


def cases(b):
    return [
        ((16, 512, 128), b.BF16, b.QParams.asym(4, 0, 15, axis=b.ALONG_T, group=64, residual=16,
                                                 scale_dtype=b.BF16, zero_dtype=b.BF16)),
        ((16, 512, 128), b.BF16, b.QParams.asym(4, 0, 15, axis=b.ALONG_C, group=64, residual=16,
                                                 scale_dtype=b.BF16, zero_dtype=b.BF16)),
        ((2, 1024, 512), b.F32, b.QParams.sym(8, axis=b.ALONG_T, group=0)),
        ((3, 77, 24), b.F32, b.QParams.sym(2, axis=b.ALONG_C, group=8)),          # generic kernels
    ]


def test_noalloc_matches_workspace_version_twice(b):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    for shape, xd, qp in cases(b):
        dt = torch.bfloat16 if xd == b.BF16 else torch.float32
        x = (torch.randn(shape, generator=g, device="cuda") * 3).to(dt)
        qt = b.quantize(x, qp)
        want = b.error_stats(x, qt)                      # the entry point with a workspace
        torch.cuda.synchronize()
        ref = want.cpu().numpy()
        for _ in range(2):                               # two calls in a row share the array
            out = torch.full((3,), -1.0, dtype=torch.float64, device="cuda")
            b.kvq_error_stats_noalloc(x, xd, qt.codes, qt.scale, qt.zero, qt.resid, qt.shape, qp, out)
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            np.testing.assert_allclose(got, ref, rtol=RTOL, atol=0)
            assert np.all(got >= 0)


def test_noalloc_rejects_shapes_beyond_the_array(b):
    """A shape whose partial sums exceed the fixed array is refused with a
    clear message before anything is launched."""
    import torch
    shape = (4096, 4096, 8)            # per-channel tiles: far more blocks than the array holds
    qp = b.QParams.sym(8, axis=b.ALONG_T, group=16)
    assert b.kvq_quantized_sizes(shape, b.BF16, qp)[4] > b.NOALLOC_SCRATCH_BYTES
    fake = 1 << 24                     # never dereferenced: the size check fails first
    out = torch.zeros(3, dtype=torch.float64, device="cuda")
    with pytest.raises(b.KvqError) as e:
        b.kvq_error_stats_noalloc(fake, b.BF16, fake, fake, None, None, shape, qp, out)
    assert e.value.status == b.EWORKSPACE
    assert "fixed" in str(e.value) and str(b.NOALLOC_SCRATCH_BYTES) in str(e.value)
