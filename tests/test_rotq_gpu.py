"""The rotation fused into per-token quantize / dequantize vs the CPU oracle.

The kernels split a row index into (slice, token) with a multiply-high
divider by T; the cases cover T = 1, small T with thousands of slices, odd T
and powers of two.

Quantize: the oracle rotates the bf16 source with its binary32 fast
transform, rounds the result to bf16 and quantizes that tensor with
oracle.quantize; codes, scales, zero points and the residual rows (rotated)
must match bit for bit.  Dequantize + inverse rotation: oracle.dequantize into
bf16, then the inverse binary32 transform rounded to bf16; bit for bit.  The
fused calls must also give what the two separate library calls give.
Every output is a guarded window (canary bytes around it must survive).
"""
import zlib

import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb, kq_of, meta_np_dtype, to_host
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def make_x(rng, shape, kind):
    if kind == "normal":
        x = W.random_kv(rng, shape)
    elif kind == "wide":        # magnitudes spanning many binades: slow quotient paths
        x = rng.standard_normal(shape) * np.exp(rng.uniform(-25, 25, shape[:2] + (1,)))
    elif kind == "ties":        # a coarse grid: many equal rotated values
        x = rng.integers(-3, 4, shape) * 0.25
    elif kind == "zeros":
        x = np.zeros(shape)
    else:
        raise ValueError(kind)
    return W.to_bf16_bits(np.asarray(x, np.float32))


def oracle_fused(xb, signs, oq):
    """The oracle's chain: binary32 rotation rounded to bf16, then quantize;
    then dequantize into bf16 and the inverse rotation rounded to bf16."""
    yb = O.rotate_fwht32(xb, O.BF16, signs, out_dtype=O.BF16)
    want = O.quantize(yb, O.BF16, oq)
    xh = O.dequantize(want, xb.shape, oq, O.BF16)
    back = O.rotate_fwht32(xh, O.BF16, signs, inverse=True, out_dtype=O.BF16)
    return want, back


def run_case(b, shape, oq, kind, seed, check_two_calls=True):
    import torch
    rng = np.random.default_rng(seed)
    xb = make_x(rng, shape, kind)
    C = shape[2]
    signs = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
    want, back = oracle_fused(xb, signs, oq)
    kq = kq_of(b, oq)
    cB, sB, zB, rB, _ = b.kvq_quantized_sizes(shape, b.BF16, kq)
    g = Guarded()
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    sd = torch.from_numpy(signs).cuda()
    codes, scale, zero, resid = g.alloc(cB), g.alloc(sB), g.alloc(zB), g.alloc(rB)
    b.kvq_rotate_quantize(x, b.BF16, shape, sd, kq, codes, scale, zero, resid)
    torch.cuda.synchronize()
    g.check("kvq_rotate_quantize")
    if cB:
        assert np.array_equal(to_host(codes), want.codes), "codes differ"
    if sB:
        assert np.array_equal(to_host(scale).view(meta_np_dtype(oq.scale_dtype)), want.scale), "scale differs"
    if zB:
        assert np.array_equal(to_host(zero).view(meta_np_dtype(oq.zero_dtype)), want.zero), "zero differs"
    if rB:
        assert np.array_equal(to_host(resid).view(np.uint16), want.resid.view(np.uint16)), "residual rows differ"
    out = g.alloc(xb.nbytes)
    b.kvq_dequantize_rotate(codes, scale, zero, resid, shape, kq, sd, out, b.BF16)
    torch.cuda.synchronize()
    g.check("kvq_dequantize_rotate")
    assert np.array_equal(to_host(out).view(np.uint16).reshape(shape), back), "dequantized rotation differs"
    if check_two_calls:
        # the same results through the two separate calls
        y = torch.empty_like(x)
        b.kvq_rotate(x, b.BF16, shape, sd, False, y, b.BF16)
        qt = b.quantize(y, kq)
        xh = b.dequantize(qt)
        z = torch.empty_like(x)
        b.kvq_rotate(xh, b.BF16, shape, sd, True, z, b.BF16)
        torch.cuda.synchronize()
        if cB:
            assert np.array_equal(to_host(qt.codes), to_host(codes)), "two calls: codes differ"
        assert np.array_equal(to_host(z).view(np.uint16), to_host(out).view(np.uint16).reshape(shape)), \
            "two calls: dequantized rotation differs"


# C, g, bits, mode (qmin, qmax) or None (symmetric), scale dtype, zero dtype, outer, T, R, kind
CASES = [
    (128, 64, 4, (0, 15), O.BF16, O.BF16, 3, 300, 16, "normal"),      # KIVI value cache format
    (128, 128, 8, None, O.F32, O.NONE, 2, 257, 0, "normal"),
    (128, 32, 2, None, O.BF16, O.NONE, 2, 100, 128, "normal"),        # all tokens in the residual window
    (128, 64, 4, (0, 15), O.BF16, O.BF16, 2, 131, 3, "wide"),
    (128, 64, 4, (0, 15), O.BF16, O.BF16, 2, 96, 0, "ties"),
    (128, 64, 8, (-128, 127), O.F32, O.I8, 2, 50, 2, "zeros"),
    (64, 64, 4, (-8, 7), O.F32, O.I8, 3, 77, 5, "normal"),
    (64, 32, 2, (0, 3), O.BF16, O.BF16, 1, 33, 0, "normal"),
    (32, 32, 8, (0, 255), O.BF16, O.F32, 2, 1000, 0, "normal"),
    (32, 32, 4, None, O.F32, O.NONE, 1, 7, 1, "wide"),
    (256, 128, 4, None, O.BF16, O.NONE, 2, 129, 1, "normal"),
    (256, 256, 8, (-128, 127), O.F32, O.F32, 1, 64, 70, "normal"),
    (256, 32, 2, (-2, 1), O.F32, O.BF16, 2, 45, 9, "wide"),
    (128, 128, 4, None, O.BF16, O.NONE, 5000, 3, 1, "normal"),      # many slices of 3 tokens
    (64, 32, 4, (0, 15), O.BF16, O.BF16, 777, 1, 0, "normal"),        # T = 1
    (128, 64, 4, (0, 15), O.BF16, O.BF16, 3, 8191, 128, "normal"),    # odd T, ragged last warp
]


@pytest.mark.parametrize("case", CASES, ids=str)
def test_rotate_quantize_matches_oracle(b, case):
    C, g, bits, qr, sd, zd, outer, T, R, kind = case
    if qr is None:
        oq = O.QParams.sym(bits, axis=O.ALONG_C, group=g, residual=R, scale_dtype=sd)
    else:
        oq = O.QParams.asym(bits, qr[0], qr[1], axis=O.ALONG_C, group=g, residual=R, scale_dtype=sd, zero_dtype=zd)
    run_case(b, (outer, T, C), oq, kind, zlib.crc32(repr(case).encode()))


def test_rotate_quantize_full_kivi_value_cache(b):
    """The KIVI value cache at full size ([64, 8192, 128] bf16, 4-bit asymmetric
    per token, groups of 64 channels, bf16 metadata, 128-token residual window),
    every output compared."""
    oq = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=128, scale_dtype=O.BF16, zero_dtype=O.BF16)
    run_case(b, (64, 8192, 128), oq, "normal", 7, check_two_calls=False)


def test_rotate_quantize_empty(b):
    oq = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=4, scale_dtype=O.BF16, zero_dtype=O.BF16)
    kq = kq_of(b, oq)
    b.kvq_rotate_quantize(None, b.BF16, (0, 5, 128), None, kq, None, None, None, None)
    b.kvq_dequantize_rotate(None, None, None, None, (4, 0, 128), kq, None, None, b.BF16)
