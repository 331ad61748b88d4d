"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Nothing here re-types the oracle's formulas.  The oracle is checked against:
worked examples and tables printed on the pages (tests/golden/, each citing
its page and section), hand-derived closed forms, invariants, special cases
that reduce to a library routine (numpy's float32 axis-0 sum, torch's bf16
rounding), and brute force on tiny inputs.  Each test names the plausible
mistake it would catch.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from kv_cache_quantization_kvq_gb300 import workloads as W


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def unpack(codes: np.ndarray, n: int, bits: int, signed: bool) -> np.ndarray:
    """Independent unpacking of the documented layout (element c in byte
    c*bits//8, lowest bits first)."""
    per = 8 // bits
    out = np.empty(n, np.int64)
    for i in range(n):
        f = (int(codes[i // per]) >> ((i % per) * bits)) & ((1 << bits) - 1)
        if signed and f >= (1 << (bits - 1)):
            f -= 1 << bits
        out[i] = f
    return out


def bf16_bits(a) -> np.ndarray:
    """bf16 rounding of float32 values by torch (a library routine)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- worked example


def test_worked_example_int4_symmetric(golden_dir):
    """Page's 4-bit example: x=[-1,-0.2,0.3,1], s=1/7 -> q=[-7,-1,2,7].
    Catches: dividing by 2^(bits-1) instead of qmax, truncation instead of
    rounding, a wrong clip range."""
    g = load(golden_dir, "worked_example_int4.json")
    x = np.array(g["x"], np.float32).reshape(1, 1, 4)
    qp = O.QParams.sym(4, axis=O.ALONG_C, group=4)
    qt = O.quantize(x, O.F32, qp)
    assert qt.scale.shape == (1,)
    assert qt.scale[0] == np.float32(1.0) / np.float32(7.0)
    assert abs(float(qt.scale[0]) - g["scale_num"] / g["scale_den"]) < 1e-7
    q = unpack(qt.codes, 4, 4, signed=True)
    assert q.tolist() == g["q"]
    xh = O.dequantize(qt, x.shape, qp, O.F32).ravel()
    want = np.array(g["x_hat_num"], np.float64) / g["x_hat_den"]
    np.testing.assert_allclose(xh, want, rtol=2e-7, atol=0)
    # the same example along the token axis (two identical channels)
    xt = np.repeat(np.array(g["x"], np.float32).reshape(1, 4, 1), 2, axis=2)
    qt2 = O.quantize(xt, O.F32, O.QParams.sym(4, axis=O.ALONG_T, group=4))
    q2 = unpack(qt2.codes, 8, 4, signed=True).reshape(4, 2)
    assert q2[:, 0].tolist() == g["q"] and q2[:, 1].tolist() == g["q"]


def test_worked_example_error_stats(golden_dir):
    """|x - x_hat| = [0, 2/35, 1/70, 0] -> max 2/35, mean 1/56, rmse sqrt(17/19600).
    Catches: a missing sqrt, dividing by N-1, max of signed error."""
    g = load(golden_dir, "worked_example_int4.json")
    x = np.array(g["x"], np.float32).reshape(1, 1, 4)
    qp = O.QParams.sym(4, axis=O.ALONG_C, group=4)
    qt = O.quantize(x, O.F32, qp)
    rmse, mx, mean = O.error_stats(x, O.F32, qt, qp)
    assert mx == pytest.approx(g["max_abs"][0] / g["max_abs"][1], rel=1e-6)
    assert mean == pytest.approx(g["mean_abs"][0] / g["mean_abs"][1], rel=1e-6)
    assert rmse == pytest.approx(math.sqrt(g["rmse_sq"][0] / g["rmse_sq"][1]), rel=1e-6)


def test_packing_convention_worked_example():
    """The documented packing of q=[-7,-1,2,7] at 4 bits: fields (q & 15) =
    [9, 15, 2, 7], low nibble first -> bytes [0xF9, 0x72]; at 2 bits the codes
    [1, -1, 0, 1] -> fields [1, 3, 0, 1] -> one byte 0b01_00_11_01."""
    x = np.array([-1, -0.2, 0.3, 1], np.float32).reshape(1, 1, 4)
    qt = O.quantize(x, O.F32, O.QParams.sym(4, axis=O.ALONG_C))
    assert qt.codes.tolist() == [0xF9, 0x72]
    x2 = np.array([1, -1, 0, 1], np.float32).reshape(1, 1, 4)
    qt2 = O.quantize(x2, O.F32, O.QParams.sym(2, axis=O.ALONG_C))
    assert qt2.codes.tolist() == [0b01001101]


# ---------------------------------------------------------------- rounding and clipping


def test_round_half_to_even_and_qmax_divisor():
    """amax 7 with qmax 7 gives s = 1 exactly, so codes are rint(x).
    Half-way cases go to the even integer (numpy's round).  Catches:
    round-half-away-from-zero, floor(x+0.5), dividing by qmax+1."""
    x = np.array([7, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5], np.float32).reshape(1, 1, 8)
    qt = O.quantize(x, O.F32, O.QParams.sym(4, axis=O.ALONG_C))
    assert qt.scale[0] == 1.0
    assert unpack(qt.codes, 8, 4, True).tolist() == [7, 2, 4, -2, -4, 0, 2, 0]


def test_true_division_not_reciprocal_multiply():
    """[FtC] §1.1 divides by the scale.  amax 3 with qmax 7 gives s = RN(3/7);
    x = 1.5*s is exact, so x/s = 1.5 exactly and rounds to the even 2.
    Multiplying by the float32 reciprocal of s gives 1.4999999 and the code 1."""
    f = np.float32
    s = f(3) / f(7)
    x1 = f(f(1.5) * s)
    assert x1 / s == f(1.5) and f(x1 * (f(1) / s)) < f(1.5)     # the trap is real
    x = np.array([3, x1, -x1, 0], np.float32).reshape(1, 1, 4)
    qt = O.quantize(x, O.F32, O.QParams.sym(4, axis=O.ALONG_C))
    assert qt.scale[0] == s
    assert unpack(qt.codes, 4, 4, True).tolist() == [7, 2, -2, 0]


def test_codes_never_exceed_qmax_with_bf16_scale():
    """With a bf16 scale, amax/s can round past qmax (up to 127.5 at INT8):
    the code must clip to qmax as an integer (no int8 wrap-around to -128)."""
    rng = np.random.default_rng(11)
    hit = 0
    for _ in range(200):
        x = rng.standard_normal((1, 64, 8)).astype(np.float32) * rng.uniform(0.1, 100)
        for bits in (8, 4, 2):
            qp = O.QParams.sym(bits, axis=O.ALONG_T, group=16, scale_dtype=O.BF16)
            qt = O.quantize(x, O.F32, qp)
            q = unpack(qt.codes, x.size, bits, True)
            qmax = (1 << (bits - 1)) - 1
            assert q.min() >= -qmax and q.max() <= qmax
            hit += int((np.abs(q) == qmax).sum())
    assert hit > 0


def test_amax_element_maps_to_qmax_fp32_scale():
    """Closed form: with a float32 scale the abs-max element of every group
    quantizes to +-qmax, and every code lies in [-qmax, qmax]."""
    rng = np.random.default_rng(3)
    for bits in (8, 4, 2):
        qmax = (1 << (bits - 1)) - 1
        x = rng.standard_normal((2, 48, 16)).astype(np.float32)
        qt = O.quantize(x, O.F32, O.QParams.sym(bits, axis=O.ALONG_T, group=16))
        q = unpack(qt.codes, x.size, bits, True).reshape(x.shape)
        for o in range(2):
            for gi in range(3):
                blk = x[o, gi * 16:(gi + 1) * 16]
                qb = q[o, gi * 16:(gi + 1) * 16]
                for c in range(16):
                    i = int(np.argmax(np.abs(blk[:, c])))
                    assert qb[i, c] == np.sign(blk[i, c]) * qmax


def test_round_trip_bound():
    """Lab line 'INT4 round-trip bound: PASS' (section '动手实验' of
    'KV cache 压缩：把历史装得更小'): for every element whose code is not
    clipped, |x - x_hat| <= s/2 (plus one float32 rounding of x/s)."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((2, 64, 32)) * 3).astype(np.float32)
    cases = [O.QParams.sym(b, axis=ax, group=g, scale_dtype=sd)
             for b in (8, 4, 2) for ax in (O.ALONG_T, O.ALONG_C) for g in (8, 32)
             for sd in (O.F32, O.BF16)]
    cases += [O.QParams.asym(4, 0, 15, axis=ax, group=16, scale_dtype=O.BF16, zero_dtype=O.BF16)
              for ax in (O.ALONG_T, O.ALONG_C)]
    cases += [O.QParams.asym(8, -128, 127, axis=O.ALONG_T, group=0)]
    for qp in cases:
        qt = O.quantize(x, O.F32, qp)
        xh = O.dequantize(qt, x.shape, qp, O.F32)
        signed = qp.mode == O.SYM or qp.qmin < 0
        q = unpack(qt.codes, x.size, qp.bits, signed).reshape(x.shape)
        s = (O.bf16_bits_to_f32(qt.scale) if qp.scale_dtype == O.BF16 else qt.scale).astype(np.float64)
        # broadcast the group scale back to elements
        if qp.axis == O.ALONG_T:
            g = qp.group or x.shape[1]
            se = np.repeat(s.reshape(2, -1, 32), g, axis=1)[:, :64]
        else:
            g = qp.group or x.shape[2]
            se = np.repeat(s.reshape(2, 64, -1), g, axis=2)[:, :, :32]
        lo = -qp.qmax if qp.mode == O.SYM else qp.qmin
        inner = (q > lo) & (q < qp.qmax)
        err = np.abs(x.astype(np.float64) - xh.astype(np.float64))
        bound = se / 2 * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -23
        assert np.all(err[inner] <= bound[inner]), qp


def test_all_zero_group_uses_range_floor():
    """[FtC] §1.1 clip at 1e-8: an all-zero group gets s = 1e-8/qmax (not a
    division by zero) and codes and x_hat equal 0."""
    x = np.zeros((1, 4, 8), np.float32)
    for bits in (8, 4, 2):
        qp = O.QParams.sym(bits, axis=O.ALONG_T)
        qmax = (1 << (bits - 1)) - 1
        qt = O.quantize(x, O.F32, qp)
        assert np.all(np.isfinite(qt.scale))
        np.testing.assert_allclose(qt.scale.astype(np.float64) * qmax, 1e-8, rtol=1e-6)
        assert not qt.codes.any()
        assert not O.dequantize(qt, x.shape, qp, O.F32).any()


def test_grid_aligned_values_round_trip_exactly():
    """x = k*s with s a power of two and k in [-qmax, qmax] (both extremes
    present) reconstructs exactly and every error statistic is 0."""
    for bits in (8, 4, 2):
        qmax = (1 << (bits - 1)) - 1
        s = 2.0 ** -3
        rng = np.random.default_rng(bits)
        k = rng.integers(-qmax, qmax + 1, size=(3, 10, 8))
        k[:, 0, :] = qmax
        k[:, 1, :] = -qmax
        x = (k * s).astype(np.float32)
        qp = O.QParams.sym(bits, axis=O.ALONG_T, group=10)
        qt = O.quantize(x, O.F32, qp)
        assert np.all(qt.scale == np.float32(s))
        assert np.array_equal(O.dequantize(qt, x.shape, qp, O.F32), x)
        assert O.error_stats(x, O.F32, qt, qp) == (0.0, 0.0, 0.0)


# ---------------------------------------------------------------- asymmetric


def test_asymmetric_hand_examples():
    """Hand-derived from [FtC] §1.2:
    x=[1,4,16], [0,15]: s=1, zp=rint(0-1)=-1, q=[0,3,15], x_hat=x.
    x=[-2,5.5,1.25,0.75], [0,15]: s=0.5, zp=4, x/s=[-4,11,2.5,1.5] ->
    rint [-4,11,2,2] -> q=[0,15,6,6], x_hat=[-2,5.5,1,1].
    Catches: a dropped zero point, a sign error in zp, zp added before rounding."""
    qp = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, zero_dtype=O.F32)
    x = np.array([1, 4, 16, 16], np.float32).reshape(1, 1, 4)
    qt = O.quantize(x, O.F32, qp)
    assert qt.scale[0] == 1.0 and qt.zero[0] == -1.0
    assert unpack(qt.codes, 4, 4, False).tolist() == [0, 3, 15, 15]
    assert np.array_equal(O.dequantize(qt, x.shape, qp, O.F32), x)

    x = np.array([-2, 5.5, 1.25, 0.75], np.float32).reshape(1, 1, 4)
    qt = O.quantize(x, O.F32, qp)
    assert qt.scale[0] == 0.5 and qt.zero[0] == 4.0
    assert unpack(qt.codes, 4, 4, False).tolist() == [0, 15, 6, 6]
    assert O.dequantize(qt, x.shape, qp, O.F32).ravel().tolist() == [-2, 5.5, 1, 1]

    # odd zero point: x=[-1.5,6,1.25]: s=0.5, zp=3, x/s=2.5 -> rint 2 -> q=5.
    # Adding zp before rounding would give rint(5.5) = 6.
    x = np.array([-1.5, 6, 1.25, 1.25], np.float32).reshape(1, 1, 4)
    qt = O.quantize(x, O.F32, qp)
    assert qt.scale[0] == 0.5 and qt.zero[0] == 3.0
    assert unpack(qt.codes, 4, 4, False).tolist() == [0, 15, 5, 5]


def test_asymmetric_int8_extremes_and_zero():
    """[FtC] §1.2 at qmin=-128, qmax=127: x=[-1, 0, 3.25]: s=4.25/255,
    -1/s = -60 -> zp = -68; the min maps to qmin, 0 maps to zp, the max to qmax."""
    qp = O.QParams.asym(8, -128, 127, axis=O.ALONG_C, zero_dtype=O.I8)
    x = np.array([-1, 0, 3.25, 0], np.float32).reshape(1, 1, 4)
    qt = O.quantize(x, O.F32, qp)
    assert qt.zero[0] == -68
    assert unpack(qt.codes, 4, 8, True).tolist() == [-128, -68, 127, -68]


def test_int8_zero_point_saturates():
    """Reading of the pages' int8 zero point: saturate, do not wrap.
    x=[10,11]: s=1/255, zp=rint(-128-2550) -> -128; codes clip to 127 and
    x_hat = (127+128)/255 = 1."""
    qp = O.QParams.asym(8, -128, 127, axis=O.ALONG_C, zero_dtype=O.I8)
    x = np.array([10, 11], np.float32).reshape(1, 1, 2)
    qt = O.quantize(x, O.F32, qp)
    assert qt.zero[0] == -128
    assert unpack(qt.codes, 2, 8, True).tolist() == [127, 127]
    np.testing.assert_allclose(O.dequantize(qt, x.shape, qp, O.F32).ravel(), [1.0, 1.0], rtol=1e-6)


def test_asymmetric_min_max_map_to_range_ends():
    """Closed form: min -> qmin and max -> qmax (within one code where both
    x/s and the zero point sit on a rounding tie); codes stay in range."""
    rng = np.random.default_rng(9)
    exact = total = 0
    for qmin, qmax, bits in ((0, 15, 4), (0, 3, 2), (-128, 127, 8), (0, 255, 8)):
        x = (rng.standard_normal((4, 32, 16)) * 2 + 0.3).astype(np.float32)
        qp = O.QParams.asym(bits, qmin, qmax, axis=O.ALONG_C, group=16, zero_dtype=O.F32)
        qt = O.quantize(x, O.F32, qp)
        q = unpack(qt.codes, x.size, bits, qmin < 0).reshape(-1, 16)
        xf = x.reshape(-1, 16)
        assert q.min() >= qmin and q.max() <= qmax
        for r in range(xf.shape[0]):
            qa, qb = q[r, np.argmin(xf[r])], q[r, np.argmax(xf[r])]
            assert abs(qa - qmin) <= 1 and abs(qb - qmax) <= 1
            exact += int(qa == qmin) + int(qb == qmax)
            total += 2
    assert exact / total > 0.99


# ---------------------------------------------------------------- axes, layout, residual


def test_axes_layout_and_residual_hand_example():
    """[KVC] KIVI: K per channel (groups along tokens), V per token (groups
    along channels).  x = [[1, 8, 0, 0], [-4, 2, 0, 0], [5, 6, 0, 0]] with R=1
    (the last token kept) at INT2 (qmax 1):
      along T: channel scales [4, 8, f, f] (f = the 1e-8 floor);
               codes rint([[.25,1],[-1,.25]]) = [[0,1],[-1,0]] (+ zeros)
      along C: token scales [8, 4]; codes rint([[.125,1],[-1,.5]]) = [[0,1],[-1,0]]
    packed 2 bits/code along C: rows -> bytes [0b0100, 0b0011]; residual =
    [5, 6, 0, 0].  Catches: transposed metadata, the wrong reduction axis, a
    residual taken from the front of the sequence."""
    x = np.array([[1, 8, 0, 0], [-4, 2, 0, 0], [5, 6, 0, 0]], np.float32).reshape(1, 3, 4)
    f = float(np.float32(1e-8))
    for axis, scales in ((O.ALONG_T, [4.0, 8.0, f, f]), (O.ALONG_C, [8.0, 4.0])):
        qp = O.QParams.sym(2, axis=axis, residual=1)
        qt = O.quantize(x, O.F32, qp)
        assert qt.scale.tolist() == pytest.approx(scales, rel=1e-7)
        assert qt.codes.tolist() == [0b0100, 0b0011]
        assert qt.resid.tolist() == [5.0, 6.0, 0.0, 0.0]
        xh = O.dequantize(qt, x.shape, qp, O.F32)
        assert xh[0, 2].tolist() == [5.0, 6.0, 0.0, 0.0]
        assert xh[0, :2].tolist() == [[0.0, 8.0, 0.0, 0.0], [-4.0, 0.0, 0.0, 0.0]] or axis == O.ALONG_C
    # along C the second token's 2 maps to rint(0.5) = 0 and its -4 to -1 -> x_hat [-4, 0]
    qp = O.QParams.sym(2, axis=O.ALONG_C, residual=1)
    xh = O.dequantize(O.quantize(x, O.F32, qp), x.shape, qp, O.F32)
    assert xh[0, :2].tolist() == [[0.0, 8.0, 0.0, 0.0], [-4.0, 0.0, 0.0, 0.0]]


def test_partial_last_group_gets_its_own_scale():
    """ceil(N/g) groups ([KVC] storage formula): T=5, g=2 along tokens gives
    groups {0,1}, {2,3}, {4}; each has its own abs-max."""
    x = np.array([1, 2, 4, 8, 16], np.float32).reshape(1, 5, 1).repeat(8, axis=2)
    qp = O.QParams.sym(8, axis=O.ALONG_T, group=2)
    qt = O.quantize(x, O.F32, qp)
    s = qt.scale.reshape(3, 8)
    np.testing.assert_allclose(s[:, 0] * 127, [2, 8, 16], rtol=1e-7)


def test_residual_counts_in_N_with_zero_error():
    """The residual window is exact and is part of N: quantizing a tensor
    whose second half is residual gives S1/N and S2/N halved (N doubled, the
    quantized half unchanged), max unchanged."""
    rng = np.random.default_rng(2)
    xa = rng.standard_normal((1, 16, 8)).astype(np.float32)
    xb = np.concatenate([xa, rng.standard_normal((1, 16, 8)).astype(np.float32)], axis=1)
    qa = O.QParams.sym(4, axis=O.ALONG_T, group=8)
    qb = O.QParams.sym(4, axis=O.ALONG_T, group=8, residual=16)
    ra = O.error_stats(xa, O.F32, O.quantize(xa, O.F32, qa), qa)
    rb = O.error_stats(xb, O.F32, O.quantize(xb, O.F32, qb), qb)
    assert rb[0] == pytest.approx(ra[0] / math.sqrt(2), rel=1e-12)
    assert rb[1] == ra[1]
    assert rb[2] == pytest.approx(ra[2] / 2, rel=1e-12)
    # everything residual -> exact
    qc = O.QParams.sym(4, axis=O.ALONG_T, residual=64)
    assert O.error_stats(xa, O.F32, O.quantize(xa, O.F32, qc), qc) == (0.0, 0.0, 0.0)


# ---------------------------------------------------------------- bf16 storage


def test_bf16_scale_rounding_matches_torch():
    """With qmax = 1 the scale is amax itself, so the stored bf16 scale is
    bf16(amax): compare with torch's float32 -> bf16 conversion, including
    exact ties (low half 0x8000) and values that round up across a binade."""
    rng = np.random.default_rng(4)
    mags = rng.standard_normal(512).astype(np.float32)
    u = mags.view(np.uint32)
    u[:64] = (u[:64] & 0xFFFF0000) | 0x8000           # exact ties
    u[64:96] = (u[64:96] & 0xFF800000) | 0x7FFFFF     # round up into next binade
    z = np.zeros_like(mags)
    x = np.stack([np.abs(mags), z, z, z], axis=1).reshape(512, 1, 4).astype(np.float32)
    qp = O.QParams.sym(2, axis=O.ALONG_C, scale_dtype=O.BF16)
    qt = O.quantize(x, O.F32, qp)
    assert np.array_equal(qt.scale, bf16_bits(np.abs(mags)))


def test_bf16_output_matches_torch_rounding_of_fp32_output():
    """Dequantizing to bf16 equals torch's bf16 rounding of the float32 x_hat."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 32, 16)).astype(np.float32)
    qp = O.QParams.sym(8, axis=O.ALONG_T, group=8)
    qt = O.quantize(x, O.F32, qp)
    f32 = O.dequantize(qt, x.shape, qp, O.F32)
    b16 = O.dequantize(qt, x.shape, qp, O.BF16)
    assert np.array_equal(b16.ravel(), bf16_bits(f32.ravel()))


def test_bf16_input_is_widened_exactly():
    """bf16 input bits widen exactly: quantizing the bf16 tensor equals
    quantizing its float32 widening (codes, scale)."""
    rng = np.random.default_rng(8)
    xb = bf16_bits(rng.standard_normal((2, 16, 16)).astype(np.float32)).reshape(2, 16, 16)
    xf = O.bf16_bits_to_f32(xb)
    qp = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=8, scale_dtype=O.BF16, zero_dtype=O.BF16)
    a, b = O.quantize(xb, O.BF16, qp), O.quantize(xf, O.F32, qp)
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.scale, b.scale)


# ---------------------------------------------------------------- sizes and ratios


def test_storage_table(golden_dir):
    """[KVC] table: INT4 + bf16 scale + bf16 zero per group of g numbers."""
    g = load(golden_dir, "storage_table_int4.json")
    N = 1 << 20
    for row in g["rows"]:
        qp = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=row["g"], scale_dtype=O.BF16,
                            zero_dtype=O.BF16)
        cB, sB, zB, rB = O.sizes((1, N // 128, 128), O.BF16, qp)
        assert (cB + sB + zB + rB) / N == row["bytes_per_number"]
        ratio = O.compression_ratio(2 * N, cB, sB, zB, rB)
        assert round(ratio, row["ratio_decimals"]) == row["ratio_vs_bf16"]


def test_exercise1_and_lab_metadata_line(golden_dir):
    """Exercise 1 / lab line: 1,048,576 bf16 numbers at INT4 g=64 -> 576 KiB, 3.556x."""
    g = load(golden_dir, "exercise1_metadata.json")
    N = g["numbers"]
    qp = O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=g["group"], scale_dtype=O.BF16,
                        zero_dtype=O.BF16)
    cB, sB, zB, rB = O.sizes((1, N // 128, 128), O.BF16, qp)
    assert cB + sB + zB + rB == g["total_bytes_KiB"] * 1024
    assert sB + zB == g["metadata_KiB"] * 1024
    assert round(O.compression_ratio(2 * N, cB, sB, zB, rB), 3) == g["ratio_printed"]


def test_residual_budget_lab_line(golden_dir):
    """Residual-window budget: one layer of K (per channel) and V (per token),
    T=8192, 8 heads, d=128, R=128, g=64 -> 32 layers = 299.500 MiB (lab line)."""
    g = load(golden_dir, "residual_budget.json")
    shape = (g["kv_heads"], g["T"], g["head_dim"])
    total = 0
    for axis in (O.ALONG_T, O.ALONG_C):
        qp = O.QParams.asym(4, 0, 15, axis=axis, group=g["group"], residual=g["residual"],
                            scale_dtype=O.BF16, zero_dtype=O.BF16)
        total += sum(O.sizes(shape, O.BF16, qp))
    assert total * g["layers"] / 2 ** 20 == g["total_MiB_printed"]


def test_cache_size_example(golden_dir):
    """Section '把节省落实到字节数': 2*32*8192*32*128*2 B = 4 GiB; the
    residual-free INT4 payload of the 8-head cache is 0.25 GiB."""
    g = load(golden_dir, "cache_size.json")
    elems = g["layers"] * g["tokens"] * g["kv_heads"] * g["head_dim"]
    assert 2 * elems * 2 == g["bf16_GiB"] * 2 ** 30
    qp = O.QParams.sym(4, axis=O.ALONG_C, group=0)
    cB, _, _, _ = O.sizes((g["layers"], g["tokens"], (g["kv_heads"] // 4) * g["head_dim"]), O.BF16, qp)
    assert 2 * cB == g["int4_payload_GiB"] * 2 ** 30


def test_symmetric_formats_omit_zero_bytes():
    """[KVC] 'symmetric schemes may omit the zero': bytes per number 0.5+2/g
    (INT4) and 0.25+2/g (INT2) with a bf16 scale only."""
    N = 128 * 1024
    for bits, base in ((4, 0.5), (2, 0.25)):
        for g in (32, 64, 128):
            qp = O.QParams.sym(bits, axis=O.ALONG_C, group=g, scale_dtype=O.BF16)
            cB, sB, zB, rB = O.sizes((1, N // 128, 128), O.BF16, qp)
            assert zB == 0 and rB == 0
            assert (cB + sB) / N == base + 2 / g


def test_token_compression_ratio_and_errors():
    """[FtC] §4: T/K, and the page's ValueError cases K<=0, K>T, T<=0."""
    assert O.token_compression_ratio(131072, 2048) == 64.0
    assert O.token_compression_ratio(5, 5) == 1.0
    for bad in ((10, 0), (10, 11), (0, 0), (-1, 1), (10, -3)):
        with pytest.raises(O.OracleError):
            O.token_compression_ratio(*bad)


def test_invalid_quantize_arguments():
    x = np.zeros((1, 4, 8), np.float32)
    bad = [O.QParams(3, O.SYM, -3, 3),                       # bits not in {2,4,8}
           O.QParams.sym(4, qmax=8),                         # qmax too large for 4 bits
           O.QParams.asym(4, 5, 5),                          # qmin >= qmax
           O.QParams.asym(4, 0, 16),                         # range does not fit
           O.QParams(4, O.SYM, -7, 7, zero_dtype=O.I8),      # symmetric with a zero buffer
           O.QParams.asym(4, 0, 15, zero_dtype=O.NONE)]      # asymmetric without one
    for qp in bad:
        with pytest.raises(O.OracleError):
            O.quantize(x, O.F32, qp)
    with pytest.raises(O.OracleError):                       # C*bits not a whole byte
        O.quantize(np.zeros((1, 4, 3), np.float32), O.F32, O.QParams.sym(4))


# ---------------------------------------------------------------- scores


def test_scores_single_row_and_integer_sums():
    hist = np.random.default_rng(1).random((3, 1, 50)).astype(np.float32)
    _, sc = O.h2o_select(hist, budget=10, window=2)
    assert np.array_equal(sc, hist[:, 0])
    ih = np.random.default_rng(2).integers(0, 1000, (2, 17, 40)).astype(np.float32)
    _, sc = O.h2o_select(ih, budget=10, window=2)
    assert np.array_equal(sc, ih.sum(axis=1, dtype=np.int64).astype(np.float32))


def test_scores_sum_rows_in_order():
    """float32 column [1, 1e8, -1e8] summed in step order gives 0 (1 is lost
    against 1e8); a reversed or re-associated order gives 1."""
    hist = np.zeros((1, 3, 4), np.float32)
    hist[0, :, 0] = [1.0, 1e8, -1e8]
    hist[0, :, 1] = [-1e8, 1e8, 1.0]
    _, sc = O.h2o_select(hist, budget=4, window=0)
    assert sc[0, 0] == 0.0 and sc[0, 1] == 1.0


def test_scores_equal_numpy_float32_axis0_sum():
    """[FtC] §3.1 sums the float32 history over axis 0 with numpy; numpy
    reduces a C-contiguous axis 0 row by row, so the bits must agree."""
    rng = np.random.default_rng(3)
    z = rng.standard_normal((4, 32, 300)) * 2
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    hist = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    _, sc = O.h2o_select(hist, budget=64, window=16)
    for h in range(4):
        assert np.array_equal(sc[h], np.sum(hist[h], axis=0))
    # softmax rows each sum to one, so the scores sum to the number of steps
    np.testing.assert_allclose(sc.sum(axis=1, dtype=np.float64), 32.0, rtol=1e-5)


def test_snapkv_score_is_mean_of_last_rows():
    """SnapKV observation score: mean of the last w rows.  Rows before the
    window must not matter; with equal rows the mean is the row itself."""
    rng = np.random.default_rng(4)
    row = rng.random(64).astype(np.float32)
    hist = np.tile(row, (1, 8, 1)).astype(np.float32)
    hist[0, :4] = 1e6                                   # outside the last-4 window
    _, sc = O.snapkv_select(hist, obs_window=4, budget=8, window=2)
    assert np.array_equal(sc[0], row)
    _, sc_all = O.snapkv_select(hist[:, 4:], obs_window=4, budget=8, window=2)
    assert np.array_equal(sc_all, sc)
    for bad in (0, 9):
        with pytest.raises(O.OracleError):
            O.snapkv_select(hist, obs_window=bad, budget=8, window=2)


# ---------------------------------------------------------------- keep-set selection


def _brute_force_keep(score, budget, window):
    """Unique subset S of the candidates [0, T-W') of size k such that every
    member outranks every non-member under (score desc, index asc); then the
    union with the recent window, sorted."""
    T = len(score)
    Wr = min(window, T)
    rs = T - Wr
    k = min(budget - Wr, rs)
    sols = []
    for S in itertools.combinations(range(rs), k):
        inS = set(S)
        ok = all(score[i] > score[j] or (score[i] == score[j] and i < j)
                 for i in S for j in range(rs) if j not in inS)
        if ok:
            sols.append(S)
    assert len(sols) == 1
    return sorted(list(sols[0]) + list(range(rs, T)))


def test_topk_union_brute_force_tiny():
    """[FtC] §3.2/§3.3: keep = TopK(score, B-W) union R_W, against brute
    force on every tiny case, with forced ties and signed zeros."""
    rng = np.random.default_rng(7)
    for trial in range(150):
        T = int(rng.integers(1, 9))
        steps = int(rng.integers(1, 3))
        if trial % 3 == 0:
            hist = rng.integers(0, 3, (1, steps, T)).astype(np.float32)   # many ties
        elif trial % 3 == 1:
            hist = rng.choice(np.array([0.0, -0.0, 1.0], np.float32), (1, 1, T))
            steps = 1
        else:
            hist = rng.random((1, steps, T)).astype(np.float32)
        budget = int(rng.integers(1, T + 3))
        window = int(rng.integers(0, budget + 1))
        keep, sc = O.h2o_select(hist, budget, window)
        assert keep[0].tolist() == _brute_force_keep(sc[0].tolist(), budget, window)


def test_keep_set_invariants_random():
    """|keep| = min(B,T); the recent window is always kept; keep is sorted
    and unique; no dropped candidate outranks a kept heavy hitter."""
    rng = np.random.default_rng(8)
    for _ in range(40):
        T = int(rng.integers(1, 400))
        hist = rng.random((2, 5, T)).astype(np.float32)
        hist[:, :, rng.integers(0, T, 5)] = 0.5                        # ties
        B = int(rng.integers(1, T + 20))
        W = int(rng.integers(0, B + 1))
        keep, sc = O.h2o_select(hist, B, W)
        for h in range(2):
            k = keep[h]
            assert len(k) == min(B, T)
            assert np.all(np.diff(k) > 0)
            Wr = min(W, T)
            assert set(range(T - Wr, T)) <= set(k.tolist())
            heavy = [i for i in k if i < T - Wr]
            dropped = [j for j in range(T - Wr) if j not in set(heavy)]
            if heavy and dropped:
                worst = min(heavy, key=lambda i: (sc[h, i], -i))
                for j in dropped:
                    assert sc[h, j] < sc[h, worst] or (sc[h, j] == sc[h, worst] and j > worst)


def test_selection_edge_cases():
    hist = np.arange(10, dtype=np.float32).reshape(1, 1, 10)
    assert O.h2o_select(hist, 20, 3)[0][0].tolist() == list(range(10))     # B >= T keeps all
    assert O.h2o_select(hist, 12, 12)[0][0].tolist() == list(range(10))    # W >= T
    assert O.h2o_select(hist, 4, 4)[0][0].tolist() == [6, 7, 8, 9]         # B == W: recent only
    assert O.h2o_select(hist, 3, 0)[0][0].tolist() == [7, 8, 9]            # W == 0: pure top-k
    assert O.h2o_select(hist[:, :, ::-1].copy(), 3, 1)[0][0].tolist() == [0, 1, 9]
    keep, _ = O.h2o_select(np.zeros((2, 3, 0), np.float32), 5, 2)           # empty sequence
    assert keep.shape == (2, 0)
    for B, W in ((3, 4), (0, 0)):                                           # W > B, B < 1
        with pytest.raises(O.OracleError):
            O.h2o_select(hist, B, W)


# ---------------------------------------------------------------- compaction


def test_compact_is_row_gather():
    rng = np.random.default_rng(9)
    kv = rng.integers(0, 65535, (3, 50, 16)).astype(np.uint16)
    keep = np.sort(rng.choice(50, (3, 7)), axis=1).astype(np.int32)
    out = O.compact(kv, keep)
    for h in range(3):
        assert np.array_equal(out[h], kv[h][keep[h]])
    with pytest.raises(O.OracleError):
        O.compact(kv, np.full((3, 2), 50, np.int32))


# ---------------------------------------------------------------- decode attention over the cache
# "KV cache 压缩：把历史装得更小" §"K 的误差会改变权重，V 的误差会改变内容":
# logit_t = q^T k_t / sqrt(d), y = sum_t a_t v_t with a = softmax(logits).


def test_attend_zero_query_is_the_mean_of_v():
    """q = 0 makes every logit 0: uniform weights, y = mean of the value rows
    (catches an unnormalised sum or a dropped row)."""
    rng = np.random.default_rng(40)
    k, v = rng.standard_normal((2, 2, 37, 16))
    y = O.attend(np.zeros((2, 3, 16)), k, v)
    for j in range(3):
        assert np.allclose(y[:, j], v.mean(axis=1), rtol=1e-13, atol=1e-15)


def test_attend_single_token_returns_its_value():
    rng = np.random.default_rng(41)
    q, k, v = rng.standard_normal((3, 4, 1, 8))
    assert np.allclose(O.attend(q, k, v)[:, 0], v[:, 0], rtol=1e-14, atol=0)


def test_attend_two_keys_sigmoid_closed_form():
    """Two keys: a_0 = 1 / (1 + exp(-(q.k0 - q.k1) / sqrt(d))) (catches a wrong
    temperature -- 1/d, no scaling -- or a transposed contraction)."""
    d = 64
    rng = np.random.default_rng(42)
    for _ in range(5):
        q = rng.standard_normal(d)
        k = rng.standard_normal((2, d))
        v = rng.standard_normal((2, d))
        a0 = 1.0 / (1.0 + math.exp(-(q @ k[0] - q @ k[1]) / math.sqrt(d)))
        want = a0 * v[0] + (1 - a0) * v[1]
        got = O.attend(q.reshape(1, 1, d), k.reshape(1, 2, d), v.reshape(1, 2, d))[0, 0]
        assert np.allclose(got, want, rtol=1e-12, atol=1e-14)


def test_attend_is_invariant_to_a_common_key_shift():
    """Adding one vector u to every key adds q.u / sqrt(d) to every logit, which
    the softmax cancels (catches a missing max subtraction that overflows, or
    weights not normalised per query)."""
    rng = np.random.default_rng(43)
    q = rng.standard_normal((2, 2, 32)) * 3
    k, v = rng.standard_normal((2, 2, 50, 32))
    u = rng.standard_normal(32) * 2000      # shifted logits near +-4000: exp overflows binary64 unless the max is taken out
    assert np.allclose(O.attend(q, k, v), O.attend(q, k + u, v), rtol=1e-9, atol=1e-11)


def test_attend_error_bounds_of_the_pages():
    """The pages' bounds: |delta logit_t| <= ||q|| ||delta k_t|| / sqrt(d), with
    equality when delta k_t is parallel to q (read off the two-key weights), and,
    for fixed weights, ||delta y|| <= max_t ||delta v_t||."""
    d = 32
    rng = np.random.default_rng(44)
    for _ in range(10):
        q = rng.standard_normal(d)
        k = rng.standard_normal((2, d))
        v = np.zeros((2, d))
        v[0, 0] = 1.0                        # y[0] = a_0: the two-key weight
        dk = q * rng.uniform(0.01, 0.3)      # delta k_0 parallel to q
        a = O.attend(q.reshape(1, 1, d), k.reshape(1, 2, d), v.reshape(1, 2, d))[0, 0, 0]
        b = O.attend(q.reshape(1, 1, d), (k + [dk, 0 * dk]).reshape(1, 2, d), v.reshape(1, 2, d))[0, 0, 0]
        dlogit = math.log(b / (1 - b)) - math.log(a / (1 - a))
        assert dlogit == pytest.approx(np.linalg.norm(q) * np.linalg.norm(dk) / math.sqrt(d), rel=1e-9)
    q = rng.standard_normal((1, 4, d))
    k, v = rng.standard_normal((2, 1, 300, d))
    dv = rng.standard_normal((1, 300, d)) * rng.uniform(0, 0.1, (1, 300, 1))
    dy = O.attend(q, k, v + dv) - O.attend(q, k, v)
    assert np.all(np.linalg.norm(dy, axis=-1) <= np.linalg.norm(dv, axis=-1).max() * (1 + 1e-12))


def test_dequantize_f64_agrees_with_the_float32_dequantizer():
    """The binary64 cache rows differ from the float32 dequantizer's x_hat by
    at most its one rounding, and the residual rows are the stored ones."""
    rng = np.random.default_rng(45)
    x = bf16_bits((rng.standard_normal((2, 300, 128)) * 2).astype(np.float32)).reshape(2, 300, 128)
    for qp in (O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=64, residual=44, scale_dtype=O.BF16, zero_dtype=O.BF16),
               O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=44, scale_dtype=O.BF16, zero_dtype=O.BF16),
               O.QParams.sym(8, axis=O.ALONG_T, group=0, residual=0),
               O.QParams.sym(2, axis=O.ALONG_C, group=32, residual=3, scale_dtype=O.BF16)):
        qt = O.quantize(x, O.BF16, qp)
        x64 = O.dequantize_f64(qt, x.shape, qp, O.BF16)
        with np.errstate(invalid="ignore"):      # its residual rows would need f32 input: not compared
            x32 = O.dequantize(qt, x.shape, qp, O.F32).astype(np.float64)
        Tq = 300 - qp.residual
        assert np.all(np.abs(x64[:, :Tq] - x32[:, :Tq]) <= np.abs(x64[:, :Tq]) * 2.0 ** -24)
        assert np.array_equal(x64[:, Tq:], O.bf16_bits_to_f32(x[:, Tq:]).astype(np.float64))


# ---------------------------------------------------------------- randomized Hadamard rotation
# KV-COBRA notes, "关键设计" item 4: an orthogonal Walsh-Hadamard matrix with
# fixed random sign flips equalises the coordinates' variances.


def test_rotate_two_channels_closed_form():
    """C = 2: the textbook 2-point transform [(a+b), (a-b)] / sqrt(2)."""
    x = np.array([[3.0, -1.25], [0.5, 0.5]])
    y = O.rotate(x, np.ones(2, np.int8))
    assert np.allclose(y, np.stack([x[:, 0] + x[:, 1], x[:, 0] - x[:, 1]], axis=1) / math.sqrt(2), rtol=1e-15)


def test_rotate_block_structure():
    """Sylvester structure: for x = [a; b], rotate_C(x) = [R(a) + R(b); R(a) - R(b)] / sqrt(2)
    with R the rotation of size C/2 (catches a sequency-ordered or transposed matrix)."""
    rng = np.random.default_rng(50)
    for C in (4, 16, 128):
        x = rng.standard_normal((3, C))
        ra = O.rotate(x[:, : C // 2], np.ones(C // 2, np.int8))
        rb = O.rotate(x[:, C // 2:], np.ones(C // 2, np.int8))
        want = np.concatenate([ra + rb, ra - rb], axis=1) / math.sqrt(2)
        assert np.allclose(O.rotate(x, np.ones(C, np.int8)), want, rtol=1e-12, atol=1e-14)


def test_rotate_is_orthogonal_and_inverted():
    """Round trips both ways are the identity and the norm is kept (catches a
    missing 1/sqrt(C), signs applied on the wrong side of the inverse)."""
    rng = np.random.default_rng(51)
    for C in (32, 128, 1024):
        x = rng.standard_normal((5, C)) * rng.uniform(0.1, 10, (5, 1))
        s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
        y = O.rotate(x, s)
        assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
        assert np.allclose(O.rotate(y, s, inverse=True), x, rtol=1e-12, atol=1e-12)
        assert np.allclose(O.rotate(O.rotate(x, s, inverse=True), s), x, rtol=1e-12, atol=1e-12)


def test_rotate_constant_vector_and_signs():
    """A constant row maps to sqrt(C) e_0; the signs act on the input:
    forward(x, s) = forward(s * x, +1)."""
    C = 64
    y = O.rotate(np.ones((1, C)), np.ones(C, np.int8))
    want = np.zeros((1, C))
    want[0, 0] = math.sqrt(C)
    assert np.allclose(y, want, atol=1e-13)
    rng = np.random.default_rng(52)
    x = rng.standard_normal((2, C))
    s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
    assert np.allclose(O.rotate(x, s), O.rotate(x * s, np.ones(C, np.int8)), rtol=1e-14, atol=1e-15)


def test_rotate_equalises_variances():
    """The page's claim: for independent coordinates with variances lam_c the
    rotated coordinates all have the mean variance, exactly:
    sum_c rotate(sqrt(lam_c) e_c)_i^2 = mean(lam) for every i."""
    C = 128
    rng = np.random.default_rng(53)
    lam = np.exp(rng.uniform(-7, 7, C))                  # spread of 1e6
    s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
    cols = O.rotate(np.diag(np.sqrt(lam)), s)           # row c = rotation of sqrt(lam_c) e_c
    assert np.allclose((cols ** 2).sum(axis=0), lam.mean(), rtol=1e-12)


# The same rotation in binary32 as the fast transform (the rotation fused into
# quantize / dequantize decides codes on binary32 values rounded to bf16).

U32 = 2.0 ** -24


def fwht_bound(x64):
    """|fast transform in binary32 - exact| <= gamma_{log2 C + 2} sum_c |x_c| / sqrt(C):
    log2(C) additions of partial sums bounded by sum |x|, one multiply by the
    rounded 1/sqrt(C) (gamma_n = n u / (1 - n u), u = 2^-24)."""
    C = x64.shape[-1]
    n = int(math.log2(C)) + 2
    return (n * U32 / (1 - n * U32)) * np.abs(x64).sum(-1, keepdims=True) / math.sqrt(C)


def test_rotate_fwht32_within_binary32_bound_of_matrix_product():
    """Against the binary64 Sylvester matrix product, both directions, both
    source dtypes (catches a dropped stage, a wrong sign or partner index)."""
    rng = np.random.default_rng(60)
    for C in (32, 64, 128, 256, 1024):
        x = (rng.standard_normal((6, C)) * np.exp(rng.uniform(-4, 4, (6, 1)))).astype(np.float32)
        s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
        for inverse in (False, True):
            want = O.rotate(x.astype(np.float64), s, inverse=inverse)
            got = O.rotate_fwht32(x, O.F32, s, inverse=inverse).astype(np.float64)
            assert np.all(np.abs(got - want) <= fwht_bound(x.astype(np.float64))), (C, inverse)
        xb = W.to_bf16_bits(x)
        x64 = O.bf16_bits_to_f32(xb).astype(np.float64)
        want = O.rotate(x64, s)
        got = O.bf16_bits_to_f32(O.rotate_fwht32(xb, O.BF16, s, out_dtype=O.BF16)).astype(np.float64)
        tol = 2.0 ** -8 * (np.abs(want) + fwht_bound(x64)) + fwht_bound(x64)   # plus the bf16 rounding
        assert np.all(np.abs(got - want) <= tol), C


def test_rotate_fwht32_exact_on_small_integers():
    """Integer inputs with |x| <= 8: every partial sum is an integer below 2^24,
    and 1/sqrt(C) is a power of two for C = 4^k, so the binary32 transform is
    exact and equals the binary64 matrix product bit for bit."""
    rng = np.random.default_rng(61)
    for C in (64, 256, 1024):
        x = rng.integers(-8, 9, (4, C)).astype(np.float32)
        s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
        for inverse in (False, True):
            got = O.rotate_fwht32(x, O.F32, s, inverse=inverse)
            want = O.rotate(x.astype(np.float64), s, inverse=inverse)
            assert np.array_equal(got.astype(np.float64), want), (C, inverse)


def test_rotate_fwht32_stage_order_worked_example():
    """Hand-derived: x = [1, 2^-24, -1, 2^-24], C = 4, no flips, scale 1/2.
    Stage h = 1: 1 + 2^-24 ties to 1; 1 - 2^-24 exact; -1 + 2^-24 exact;
    -1 - 2^-24 ties to -1, so v = [1, 1 - 2^-24, -(1 - 2^-24), -1].
    Stage h = 2: 1 - (1 - 2^-24) = 2^-24; (1 - 2^-24) - 1 = -2^-24;
    1 + (1 - 2^-24) = 2 - 2^-24 ties to 2, twice.  Times 1/2:
    [2^-25, -2^-25, 1, 1].  (Stage h = 2 first would give the exact
    [2^-24, -2^-24, 1, 1], so this pins the stage order.)"""
    x = np.array([[1.0, 2.0 ** -24, -1.0, 2.0 ** -24]], np.float32)
    got = O.rotate_fwht32(x, O.F32, np.ones(4, np.int8))
    assert np.array_equal(got, np.array([[2.0 ** -25, -2.0 ** -25, 1.0, 1.0]], np.float32))
    exact = O.rotate(x.astype(np.float64), np.ones(4, np.int8))
    assert np.array_equal(exact, np.array([[2.0 ** -24, -2.0 ** -24, 1.0, 1.0]]))


def test_rotate_fwht32_round_trip_and_bf16_rounding():
    """Inverse after forward returns x within twice the bound; a bf16 output
    is the nearest-even bf16 of the binary32 output."""
    rng = np.random.default_rng(62)
    C = 128
    x = rng.standard_normal((5, C)).astype(np.float32)
    s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
    y = O.rotate_fwht32(x, O.F32, s)
    back = O.rotate_fwht32(y, O.F32, s, inverse=True).astype(np.float64)
    assert np.all(np.abs(back - x) <= 2 * fwht_bound(x.astype(np.float64)) + 1e-6 * np.abs(x))
    yb = O.rotate_fwht32(x, O.F32, s, out_dtype=O.BF16)
    assert np.array_equal(yb, W.to_bf16_bits(y))
