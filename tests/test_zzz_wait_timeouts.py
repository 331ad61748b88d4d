"""No bounded wait of the library's kernels gave up (kvq_wait_timeouts).

Every wait of the staged, warp-specialised and cluster kernels on an
asynchronous copy (an mbarrier phase) polls a bounded number of times; one that
runs out records itself in a device counter and its kernel leaves its loop,
leaving its outputs undefined.  Collected after every other test, so in a full run the count
covers the whole suite; it first runs each kernel family with bounded waits
once, so that it also means something on its own.
"""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_quantization_kvq_gb300 import build
    build()
    from kv_cache_quantization_kvq_gb300 import binding
    return binding


def test_no_bounded_wait_gave_up(b):
    import torch
    g = torch.Generator(device="cuda").manual_seed(9)
    x = torch.randn((8, 1024, 128), generator=g, device="cuda").to(torch.bfloat16)
    kivi_k = b.QParams.asym(4, 0, 15, axis=b.ALONG_T, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
    kivi_v = b.QParams.asym(4, 0, 15, axis=b.ALONG_C, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
    long_k = b.QParams.sym(8, axis=b.ALONG_T, group=0)              # one group over all tokens: clusters
    for qp in (kivi_k, kivi_v, long_k):
        qt = b.quantize(x, qp)
        b.dequantize(qt)
        b.error_stats(x, qt)
    assert b.kvq_wait_timeouts() == 0
