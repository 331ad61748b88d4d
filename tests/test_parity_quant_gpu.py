"""CUDA quantize / dequantize / error statistics vs the CPU oracle.

Both sides consume the same seeded host buffer.  Codes, packed bytes,
scales, zero points and residual bytes must be bit-exact; the dequantized
tensor must match the oracle bit for bit as well (stricter than the 1e-6
relative bar, since both sides perform the same IEEE operations); the error
statistics must agree within 1e-5 relative.
"""
import itertools
import zlib

import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb, kq_of, meta_np_dtype, to_device, to_host
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STATS_RTOL = 1e-5


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def make_input(rng, shape, x_dtype, kind="normal"):
    outer, T, C = shape
    if kind == "normal":
        x = W.random_kv(rng, shape) if outer * T * C else np.zeros(shape, np.float32)
    elif kind == "zeros":
        x = np.zeros(shape, np.float32)
    elif kind == "ties":       # values on a half-step grid of a power-of-two scale
        x = (rng.integers(-15, 16, shape) / 2.0 * 0.125).astype(np.float32)
    elif kind == "wide":       # magnitudes spanning many binades
        x = (rng.standard_normal(shape) * np.exp(rng.uniform(-30, 30, shape))).astype(np.float32)
    elif kind == "const":
        x = np.full(shape, 1.5, np.float32)
    else:
        raise ValueError(kind)
    return W.to_bf16_bits(x) if x_dtype == O.BF16 else x


def check_case(b, xin, x_dtype, oq, offset=0):
    """Run one case on both sides and compare.  offset > 0 shifts every
    device buffer off 16-byte alignment to exercise the generic kernels.
    Every buffer a call writes is a guarded window: canary bytes before and
    after it must be unchanged after each call (no stray stores)."""
    import torch
    shape = xin.shape
    want = O.quantize(xin, x_dtype, oq)
    kq = kq_of(b, oq)
    cB, sB, zB, rB, wB = b.kvq_quantized_sizes(shape, x_dtype, kq)
    es = 2 if x_dtype == O.BF16 else 4
    g = Guarded()

    def buf(n, off=offset):
        return g.alloc(n, off)

    xraw = buf(xin.nbytes)
    if xin.nbytes:
        xraw.copy_(torch.from_numpy(np.ascontiguousarray(xin).view(np.uint8).ravel()).cuda())
    codes, scale, zero, resid, ws = buf(cB), buf(sB), buf(zB), buf(rB), buf(wB, 0)
    b.kvq_quantize(xraw, x_dtype, shape, kq, codes, scale, zero, resid, ws, wB)
    torch.cuda.synchronize()
    g.check("kvq_quantize")
    if cB:
        assert np.array_equal(to_host(codes), want.codes), "codes differ"
    if sB:
        assert np.array_equal(to_host(scale).view(meta_np_dtype(oq.scale_dtype)), want.scale), "scale differs"
    if zB:
        assert np.array_equal(to_host(zero).view(meta_np_dtype(oq.zero_dtype)), want.zero), "zero differs"
    if rB:
        assert np.array_equal(to_host(resid).view(want.resid.dtype), want.resid), "residual differs"

    # dequantize into the source dtype (required when a residual exists) and,
    # without residual, into the other dtype as well
    out_dtypes = [x_dtype] if oq.residual else [O.F32, O.BF16]
    for od in out_dtypes:
        ref = O.dequantize(want, shape, oq, od)
        ob = buf(ref.nbytes)
        b.kvq_dequantize(codes, scale, zero, resid, shape, kq, ob, od)
        torch.cuda.synchronize()
        g.check("kvq_dequantize")
        if ref.size:
            got = to_host(ob).view(ref.dtype).reshape(shape)
            assert np.array_equal(got, ref), f"dequantized values differ (out dtype {od})"

    if xin.size:
        rmse, mx, mean = O.error_stats(xin, x_dtype, want, oq)
        sw = buf(wB, 0)
        out = g.alloc(24).view(torch.float64)
        b.kvq_error_stats(xraw, x_dtype, codes, scale, zero, resid, shape, kq, out, sw, wB)
        torch.cuda.synchronize()
        g.check("kvq_error_stats")
        gs = out.cpu().numpy()
        for got, ref, name in ((gs[0], rmse, "rmse"), (gs[1], mx, "max"), (gs[2], mean, "mean")):
            assert got == pytest.approx(ref, rel=STATS_RTOL, abs=1e-30), name


def sym(bits, **kw):
    return O.QParams.sym(bits, **kw)


def asym_ranges(bits):
    if bits == 8:
        return [(-128, 127), (0, 255)]
    return [(0, (1 << bits) - 1), (-(1 << (bits - 1)), (1 << (bits - 1)) - 1)]


# ---------------------------------------------------------------- along C (per token)

ALONG_C_CASES = []
for bits, g, xd in itertools.product((8, 4, 2), (8, 32, 64, 128, 0), (O.BF16, O.F32)):
    ALONG_C_CASES.append(("sym", bits, g, xd, O.BF16 if g % 64 == 0 else O.F32))
    for rng_ in asym_ranges(bits):
        ALONG_C_CASES.append(("asym", bits, g, xd, rng_))


@pytest.mark.parametrize("case", ALONG_C_CASES, ids=str)
def test_along_c_fast(b, case):
    mode, bits, g, xd, extra = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    shape = (3, 77, 128)
    xin = make_input(rng, shape, xd)
    if mode == "sym":
        oq = sym(bits, axis=O.ALONG_C, group=g, residual=9, scale_dtype=extra)
    else:
        oq = O.QParams.asym(bits, *extra, axis=O.ALONG_C, group=g, residual=9, scale_dtype=O.BF16,
                            zero_dtype=O.BF16 if bits < 8 else O.I8)
    check_case(b, xin, xd, oq)


@pytest.mark.parametrize("C,g", [(256, 256), (512, 64), (2048, 128), (16, 8), (8, 8)])
def test_along_c_wide_and_narrow_rows(b, C, g):
    rng = np.random.default_rng(C + g)
    xin = make_input(rng, (2, 33, C), O.BF16)
    check_case(b, xin, O.BF16, sym(4, axis=O.ALONG_C, group=g, scale_dtype=O.BF16))
    check_case(b, xin, O.BF16, O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=g, residual=5,
                                               scale_dtype=O.BF16, zero_dtype=O.BF16))


@pytest.mark.parametrize("C,g", [(24, 8), (96, 32), (128, 12), (40, 40), (64, 3)])
def test_along_c_generic_shapes(b, C, g):
    """C/8 not a power of two, g not a multiple of 8, partial last group."""
    rng = np.random.default_rng(C * 7 + g)
    for xd in (O.BF16, O.F32):
        xin = make_input(rng, (2, 19, C), xd)
        check_case(b, xin, xd, sym(8, axis=O.ALONG_C, group=g, residual=3))
        check_case(b, xin, xd, O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=g, scale_dtype=O.BF16,
                                               zero_dtype=O.BF16))


# ---------------------------------------------------------------- along T (per channel)

ALONG_T_CASES = []
for bits, g, xd in itertools.product((8, 4, 2), (16, 64, 128, 200, 0), (O.BF16, O.F32)):
    ALONG_T_CASES.append(("sym", bits, g, xd, None))
    for rng_ in asym_ranges(bits):
        ALONG_T_CASES.append(("asym", bits, g, xd, rng_))


@pytest.mark.parametrize("case", ALONG_T_CASES, ids=str)
def test_along_t_fast(b, case):
    """Register tile (g <= 128) and the long-group two-pass path (g > 128),
    several channel blocks (C = 256) and a ragged last group."""
    mode, bits, g, xd, qrange = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    shape = (2, 301, 256)
    xin = make_input(rng, shape, xd)
    if mode == "sym":
        oq = sym(bits, axis=O.ALONG_T, group=g, residual=13, scale_dtype=O.BF16 if g == 64 else O.F32)
    else:
        qmin, qmax = qrange
        oq = O.QParams.asym(bits, qmin, qmax, axis=O.ALONG_T, group=g, residual=13,
                            scale_dtype=O.BF16, zero_dtype=(O.BF16, O.I8, O.F32)[g % 3])
    check_case(b, xin, xd, oq)


# Long groups along T (one scale per channel over hundreds to thousands of
# tokens), bf16 sources: the cluster kernel, where 1 to 16 CTAs share one
# group of 64 channels, one cluster per unit.  Groups of up to 2048 tokens:
# ceil(group / 512) CTAs with every row in shared memory; longer groups:
# ceil(group / 1024) CTAs with 512 rows in shared memory and the rest in
# registers (2049 tokens: 171 register rows per CTA, a ragged register tail).
# Groups beyond 8192 tokens take the two-pass path through the workspace.
# Ragged last groups (some CTAs of a cluster get no rows), residual windows,
# several channel blocks, and many more units than resident clusters.
LONG_T_CASES = [
    # bits, mode (qmin, qmax) or None, g, T, R, C, kind, outer
    (8, None, 0, 4100, 4, 128, "normal", 2),
    (8, None, 0, 8192, 0, 192, "normal", 2),
    (4, (0, 15), 1000, 2600, 7, 128, "normal", 2),
    (2, None, 3000, 6100, 0, 64, "normal", 2),
    (4, None, 5000, 5100, 50, 128, "wide", 2),
    (8, (-128, 127), 700, 1500, 3, 64, "const", 2),
    (4, (-8, 7), 2048, 4096, 0, 64, "ties", 2),
    (8, (0, 255), 0, 9000, 0, 64, "normal", 2),
    (8, (0, 255), 600, 1300, 0, 2048, "normal", 8),
    (8, None, 0, 8192, 0, 512, "normal", 4),
    (8, None, 2049, 4200, 5, 128, "wide", 3),
    (4, (0, 15), 2100, 2101, 0, 64, "ties", 2),
]


@pytest.mark.parametrize("case", LONG_T_CASES, ids=str)
def test_along_t_long_groups(b, case):
    bits, qr, g, T, R, C, kind, outer = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    xin = make_input(rng, (outer, T, C), O.BF16, kind)
    if qr is None:
        oq = sym(bits, axis=O.ALONG_T, group=g, residual=R, scale_dtype=O.F32 if bits == 8 else O.BF16)
    else:
        oq = O.QParams.asym(bits, qr[0], qr[1], axis=O.ALONG_T, group=g, residual=R,
                            scale_dtype=O.F32 if qr[0] < 0 else O.BF16, zero_dtype=O.I8 if qr[0] < 0 else O.BF16)
    check_case(b, xin, O.BF16, oq)


@pytest.mark.parametrize("C", [8, 24, 136])
def test_along_t_partial_channel_block(b, C):
    rng = np.random.default_rng(C)
    xin = make_input(rng, (3, 90, C), O.BF16)
    check_case(b, xin, O.BF16, sym(4, axis=O.ALONG_T, group=32, scale_dtype=O.BF16))
    check_case(b, xin, O.BF16, sym(8, axis=O.ALONG_T, group=0, residual=4))


# head_dim 128 with bf16 input: the warp-specialised group-tile kernel (g in
# {16, 32, 64}) and the block-tile kernel (other g <= 64), for every metadata
# layout they specialise (bf16 scale + zero, f32 scale + int8 zero, bf16 or
# f32 scale alone); ragged last quantized group, ragged residual tile.
HD128_T_CASES = []
for bits, g in itertools.product((8, 4, 2), (16, 32, 64, 48)):
    HD128_T_CASES.append(("sym", bits, g, O.BF16, O.NONE, None))
    HD128_T_CASES.append(("sym", bits, g, O.F32, O.NONE, None))
    for qr in asym_ranges(bits):
        HD128_T_CASES.append(("asym", bits, g, O.BF16, O.BF16, qr))
        HD128_T_CASES.append(("asym", bits, g, O.F32, O.I8, qr))


@pytest.mark.parametrize("case", HD128_T_CASES, ids=str)
def test_along_t_head_dim_128(b, case):
    mode, bits, g, sdt, zdt, qr = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    xin = make_input(rng, (3, 301, 128), O.BF16)
    if mode == "sym":
        oq = sym(bits, axis=O.ALONG_T, group=g, residual=13, scale_dtype=sdt)
    else:
        oq = O.QParams.asym(bits, qr[0], qr[1], axis=O.ALONG_T, group=g, residual=13, scale_dtype=sdt,
                            zero_dtype=zdt)
    check_case(b, xin, O.BF16, oq)


@pytest.mark.parametrize("kind", ["zeros", "ties", "wide", "const"])
@pytest.mark.parametrize("T,R", [(200, 0), (150, 64), (40, 128), (64, 70)])
def test_along_t_head_dim_128_values_and_lengths(b, kind, T, R):
    """Value kinds that force the IEEE-division fallback inside a tile
    ("wide"), exact ties, constant groups; no residual, a residual shorter
    than, equal to and longer than one group tile."""
    rng = np.random.default_rng(T * 7 + R + len(kind))
    xin = make_input(rng, (2, T, 128), O.BF16, kind)
    for oq in (O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=64, residual=R, scale_dtype=O.BF16,
                              zero_dtype=O.BF16),
               O.QParams.asym(2, -2, 1, axis=O.ALONG_T, group=32, residual=R, zero_dtype=O.I8),
               sym(8, axis=O.ALONG_T, group=16, residual=R, scale_dtype=O.BF16)):
        check_case(b, xin, O.BF16, oq)


# head_dim 128 with bf16 input, groups along C: the warp-specialised row
# kernel (g in {32, 64, 128}) for every metadata layout it specialises, plus
# g = 16 (the other kernels); token counts that leave a ragged last chunk of
# 32 rows and chunks that straddle the residual window and the next head.
HD128_C_CASES = []
for bits, g in itertools.product((8, 4, 2), (32, 64, 128, 16)):
    HD128_C_CASES.append(("sym", bits, g, O.BF16, O.NONE, None))
    HD128_C_CASES.append(("sym", bits, g, O.F32, O.NONE, None))
    for qr in asym_ranges(bits):
        HD128_C_CASES.append(("asym", bits, g, O.BF16, O.BF16, qr))
        HD128_C_CASES.append(("asym", bits, g, O.F32, O.I8, qr))


@pytest.mark.parametrize("case", HD128_C_CASES, ids=str)
def test_along_c_head_dim_128(b, case):
    mode, bits, g, sdt, zdt, qr = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    xin = make_input(rng, (3, 301, 128), O.BF16)
    if mode == "sym":
        oq = sym(bits, axis=O.ALONG_C, group=g, residual=13, scale_dtype=sdt)
    else:
        oq = O.QParams.asym(bits, qr[0], qr[1], axis=O.ALONG_C, group=g, residual=13, scale_dtype=sdt,
                            zero_dtype=zdt)
    check_case(b, xin, O.BF16, oq)


@pytest.mark.parametrize("kind", ["zeros", "ties", "wide", "const"])
@pytest.mark.parametrize("T,R", [(200, 0), (45, 64), (33, 1)])
def test_along_c_head_dim_128_values_and_lengths(b, kind, T, R):
    rng = np.random.default_rng(T * 11 + R + len(kind))
    xin = make_input(rng, (2, T, 128), O.BF16, kind)
    for oq in (O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=R, scale_dtype=O.BF16,
                              zero_dtype=O.BF16),
               O.QParams.asym(2, -2, 1, axis=O.ALONG_C, group=32, residual=R, zero_dtype=O.I8),
               sym(8, axis=O.ALONG_C, group=128, residual=R, scale_dtype=O.BF16)):
        check_case(b, xin, O.BF16, oq)


# ---------------------------------------------------------------- edge cases


@pytest.mark.parametrize("kind", ["zeros", "ties", "wide", "const"])
def test_value_edge_cases(b, kind):
    rng = np.random.default_rng(len(kind))
    for xd in (O.BF16, O.F32):
        xin = make_input(rng, (2, 40, 64), xd, kind)
        for oq in (sym(4, axis=O.ALONG_C, group=32, scale_dtype=O.BF16),
                   sym(8, axis=O.ALONG_T, group=16),
                   sym(2, axis=O.ALONG_T, group=0),
                   O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=16, scale_dtype=O.BF16, zero_dtype=O.BF16),
                   O.QParams.asym(8, -128, 127, axis=O.ALONG_C, group=64, zero_dtype=O.I8)):
            check_case(b, xin, xd, oq)


@pytest.mark.parametrize("shape,R", [((1, 1, 8), 0), ((1, 1, 8), 1), ((2, 5, 16), 5), ((2, 5, 16), 100),
                                     ((0, 5, 16), 2), ((2, 0, 16), 2), ((1, 129, 8), 1)])
def test_degenerate_shapes(b, shape, R):
    """Single token, everything residual, empty outer / sequence."""
    rng = np.random.default_rng(sum(shape) + R)
    for xd in (O.BF16, O.F32):
        xin = make_input(rng, shape, xd)
        for axis in (O.ALONG_T, O.ALONG_C):
            check_case(b, xin, xd, sym(4, axis=axis, group=8, residual=R))
            check_case(b, xin, xd, O.QParams.asym(8, -128, 127, axis=axis, group=0, residual=R))


@pytest.mark.parametrize("offset", [4, 8, 12])
def test_unaligned_buffers_take_generic_path(b, offset):
    rng = np.random.default_rng(offset)
    xin = make_input(rng, (2, 50, 128), O.BF16)
    for oq in (sym(4, axis=O.ALONG_C, group=32, residual=6, scale_dtype=O.BF16),
               sym(8, axis=O.ALONG_T, group=64, residual=6),
               O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=0, scale_dtype=O.BF16, zero_dtype=O.BF16)):
        check_case(b, xin, O.BF16, oq, offset=offset)


def test_tiny_config_three_quantizers(b):
    """The tiny workload: fp32 [256, 128] with 4 outlier channels; symmetric
    INT8 per channel, asymmetric INT8 per channel, symmetric INT4 in groups of
    32 tokens per channel; compression ratios with metadata."""
    x, _ = W.tiny_inputs(0)
    cases = [(sym(8, axis=O.ALONG_T, group=0), 131072 / (32768 + 512)),
             (O.QParams.asym(8, -128, 127, axis=O.ALONG_T, group=0, zero_dtype=O.I8), 131072 / (32768 + 512 + 128)),
             (sym(4, axis=O.ALONG_T, group=32), 131072 / (16384 + 4096))]
    for oq, cr in cases:
        check_case(b, x, O.F32, oq)
        kq = kq_of(b, oq)
        cB, sB, zB, rB, _ = b.kvq_quantized_sizes(x.shape, b.F32, kq)
        assert b.kvq_compression_ratio(x.nbytes, cB, sB, zB, rB) == pytest.approx(cr, rel=1e-12)
