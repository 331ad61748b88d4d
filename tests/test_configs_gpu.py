"""Parity at the workloads' full sizes, through the same C-ABI calls and
launch configurations the benchmark times.

Where the oracle finishes in seconds the whole output is compared
(KIVI INT4, H2O / SnapKV + compaction); otherwise sampled [outer] slices are
compared element by element (each slice is an independent set of groups, so
the oracle computes it alone) and size-independent properties are checked on
the full output (code range, abs-max element -> +-qmax, statistics that
combine exactly across slices).
"""
import math

import numpy as np
import pytest

import oracle as O
from gpu_util import kb, kq_of, meta_np_dtype, to_host
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu
STATS_RTOL = 1e-5


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def compare_slice(b, x_host, qt, oq, lo, hi):
    """Oracle on outer slices [lo, hi) vs the GPU buffers of the full tensor
    (only the slice's bytes leave the device)."""
    outer, T, C = x_host.shape
    xs = np.ascontiguousarray(x_host[lo:hi])
    want = O.quantize(xs, O.BF16, oq)
    n = hi - lo
    cpo, spo = want.codes.size // n, want.scale.size // n
    assert np.array_equal(to_host(qt.codes[lo * cpo:hi * cpo]), want.codes), "codes differ"
    sB = np.dtype(meta_np_dtype(oq.scale_dtype)).itemsize
    got_s = to_host(qt.scale[lo * spo * sB:hi * spo * sB]).view(meta_np_dtype(oq.scale_dtype))
    assert np.array_equal(got_s, want.scale), "scales differ"
    if want.zero.size:
        zB = np.dtype(meta_np_dtype(oq.zero_dtype)).itemsize
        got_z = to_host(qt.zero[lo * spo * zB:hi * spo * zB]).view(meta_np_dtype(oq.zero_dtype))
        assert np.array_equal(got_z, want.zero), "zeros differ"
    if want.resid.size:
        rpo = want.resid.size // n
        assert np.array_equal(to_host(qt.resid[lo * rpo * 2:hi * rpo * 2]).view(np.uint16), want.resid)
    return want, xs


def _slice_vs(b, xs, qt, oq, lo):
    """Like compare_slice for one outer slice whose host copy xs is [1, T, C]."""
    want = O.quantize(xs, O.BF16, oq)
    cpo, spo = want.codes.size, want.scale.size
    assert np.array_equal(to_host(qt.codes[lo * cpo:(lo + 1) * cpo]), want.codes), "codes differ"
    sB = np.dtype(meta_np_dtype(oq.scale_dtype)).itemsize
    got_s = to_host(qt.scale[lo * spo * sB:(lo + 1) * spo * sB]).view(meta_np_dtype(oq.scale_dtype))
    assert np.array_equal(got_s, want.scale), "scales differ"
    return want, xs


def test_kivi_int4_full(b):
    """KIVI INT4: batch 8, 8 KV heads, T 8192, d 128, bf16; K per channel
    (g 64 tokens), V per token (g 64 channels), asymmetric [0, 15], bf16
    scale + zero, 128-token residual.  Whole outputs compared."""
    import torch
    K, V = W.kivi_kv("cuda", seed=2)
    shape = (64, 8192, 128)
    total = 0
    for x, axis in ((K, O.ALONG_T), (V, O.ALONG_C)):
        oq = O.QParams.asym(4, 0, 15, axis=axis, group=64, residual=128, scale_dtype=O.BF16, zero_dtype=O.BF16)
        kq = kq_of(b, oq)
        qt = b.quantize(x.view(shape), kq)
        xh = b.dequantize(qt)
        st = b.error_stats(x.view(shape), qt)
        torch.cuda.synchronize()
        xhost = to_host(x).reshape(shape)
        want, _ = compare_slice(b, xhost, qt, oq, 0, 64)
        assert np.array_equal(to_host(xh).reshape(shape), O.dequantize(want, shape, oq, O.BF16))
        ref = O.error_stats(xhost, O.BF16, want, oq)
        np.testing.assert_allclose(st.cpu().numpy(), ref, rtol=STATS_RTOL)
        total += sum(b.kvq_quantized_sizes(shape, b.BF16, kq)[:4])
    # K + V per layer vs bf16: the residual-budget reading (3.4190x)
    assert 2 * 2 * 64 * 8192 * 128 / total == pytest.approx(33554432 * 8 / (9814016 * 8), rel=1e-12)
    assert round(2 * 2 * 64 * 8192 * 128 / total, 4) == 3.4190


def test_fullmodel_int8_per_channel(b):
    """Symmetric INT8 per channel over a 32-layer cache [32, 8192, 32*128]
    (K and V, ~4.3 GB), fp32 scale, group = all 8192 tokens, through the
    same whole-tensor calls the benchmark times.  Layers 0, 17 and 31 of the
    quantize and of the one whole-tensor dequantize are compared with the
    oracle element by element; the code range and the +-127 abs-max code are
    checked everywhere.  The whole-tensor statistics must equal the exact
    combination of per-layer sums in which layers 0, 17 and 31 come from the
    oracle and the other 29 from the GPU's per-layer statistics (which are
    themselves checked against the oracle on the three sampled layers)."""
    import torch
    K, V = W.fullmodel_kv("cuda", seed=3)
    L, T, C = 32, 8192, 4096
    shape = (L, T, C)
    n_l = T * C
    sampled = (0, 17, 31)
    oq = O.QParams.sym(8, axis=O.ALONG_T, group=0)
    kq = kq_of(b, oq)
    for x in (K, V):
        qt = b.quantize(x, kq)
        xh = b.dequantize(qt)                                  # one call over all 32 layers
        st = b.error_stats(x, qt)
        torch.cuda.synchronize()
        codes = qt.codes.view(torch.int8).view(shape)
        assert int(codes.min()) >= -127 and int(codes.max()) <= 127
        amax_code = codes.abs().amax(dim=1)                    # per (layer, channel)
        assert bool((amax_code == 127).all()), "abs-max element must map to +-127"
        del codes, amax_code
        ref_stats = {}
        for l in sampled:
            xs = to_host(x[l:l + 1]).reshape(1, T, C)
            want = O.quantize(xs, O.BF16, oq)
            assert np.array_equal(to_host(qt.codes[l * n_l:(l + 1) * n_l]), want.codes), f"codes of layer {l}"
            assert np.array_equal(to_host(qt.scale[l * C * 4:(l + 1) * C * 4]).view(np.float32), want.scale), \
                f"scales of layer {l}"
            got = to_host(xh[l:l + 1]).reshape(1, T, C)
            assert np.array_equal(got, O.dequantize(want, (1, T, C), oq, O.BF16)), f"dequantized layer {l}"
            ref_stats[l] = O.error_stats(xs, O.BF16, want, oq)
            del xs, want, got
        # statistics: per-layer sums, the sampled layers from the oracle
        s1 = s2 = mx = 0.0
        ws = torch.empty(b.kvq_quantized_sizes((1, T, C), b.BF16, kq)[4], dtype=torch.uint8, device="cuda")
        for l in range(L):
            sub = b.Quantized(qt.codes[l * n_l:(l + 1) * n_l], qt.scale[l * C * 4:(l + 1) * C * 4], qt.zero,
                              qt.resid, (1, T, C), kq, b.BF16)
            r = b.error_stats(x[l:l + 1], sub, workspace=ws).cpu().numpy()
            if l in ref_stats:
                np.testing.assert_allclose(r, ref_stats[l], rtol=STATS_RTOL)
                r = np.asarray(ref_stats[l])
            s2 += r[0] ** 2 * n_l
            s1 += r[2] * n_l
            mx = max(mx, r[1])
        full = st.cpu().numpy()
        N = L * n_l
        np.testing.assert_allclose(full, [math.sqrt(s2 / N), mx, s1 / N], rtol=STATS_RTOL)
        cB, sB, zB, rB, _ = b.kvq_quantized_sizes(shape, b.BF16, kq)
        assert round(b.kvq_compression_ratio(2 * L * T * C, cB, sB, zB, rB), 5) == 1.99902
        del qt, st, xh


@pytest.mark.parametrize("bits", [4, 2])
def test_sweep_per_token(b, bits):
    """Batch 16, 8 heads, T 32768, d 128, N(0,1) with 1 % outliers x20;
    symmetric INT4 / INT2 per token with g in {32, 64, 128} and a bf16 scale.
    Three [outer] slices compared with the oracle; bytes per number checked
    against 0.5 + 2/g (INT4) and 0.25 + 2/g (INT2)."""
    import torch
    K, V = W.sweep_kv("cuda", seed=4)
    shape = (128, 32768, 128)
    qmax = (1 << (bits - 1)) - 1
    for g in (32, 64, 128):
        oq = O.QParams.sym(bits, axis=O.ALONG_C, group=g, scale_dtype=O.BF16)
        kq = kq_of(b, oq)
        cB, sB, zB, rB, _ = b.kvq_quantized_sizes(shape, b.BF16, kq)
        N = 128 * 32768 * 128
        assert (cB + sB) / N == bits / 8 + 2 / g and zB == rB == 0
        for x in (K, V):
            qt = b.quantize(x, kq)
            xh = b.dequantize(qt)
            torch.cuda.synchronize()
            for lo in (0, 77, 127):
                xhost = to_host(x[lo:lo + 1]).reshape(1, 32768, 128)
                want, xs = _slice_vs(b, xhost, qt, oq, lo)
                got = to_host(xh[lo:lo + 1]).reshape(1, 32768, 128)
                assert np.array_equal(got, O.dequantize(want, xs.shape, oq, O.BF16))
            del qt, xh


def test_eviction_full(b):
    """32 heads, history fp32 [64, 131072] with 256 planted heavy hitters,
    B 2048, W 128; H2O and SnapKV (mean of the last 32 steps); compaction of
    bf16 K/V [32, 131072, 128].  Whole outputs compared."""
    import torch
    hist, K, V = W.eviction_inputs("cuda", seed=5)
    hh = hist.cpu().numpy()
    for obs in (None, 32):
        if obs is None:
            keep, scores = b.h2o_select(hist, 2048, 128)
            ok, osc = O.h2o_select(hh, 2048, 128)
        else:
            keep, scores = b.snapkv_select(hist, obs, 2048, 128)
            ok, osc = O.snapkv_select(hh, obs, 2048, 128)
        torch.cuda.synchronize()
        assert np.array_equal(scores.cpu().numpy().view(np.uint32), osc.view(np.uint32))
        assert np.array_equal(keep.cpu().numpy(), ok)
        for x in (K, V):
            out = b.compact(x, keep)
            torch.cuda.synchronize()
            xh = to_host(x)
            assert np.array_equal(to_host(out), O.compact(xh, ok))
        # the planted heavy hitters are found
        assert keep.shape == (32, 2048)
    assert b.kvq_token_compression_ratio(131072, 2048) == 64.0
