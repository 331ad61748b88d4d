"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library must load and export every entry point include/kvq.h declares;
the host-only size / ratio functions must agree with the oracle; every
argument check must reject bad input before anything reaches the GPU (the
pages' ValueError cases and the documented contract).
"""
import itertools
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kb():
    from kv_cache_quantization_kvq_gb300 import build
    build()
    from kv_cache_quantization_kvq_gb300 import binding
    return binding


def declared_symbols():
    with open(os.path.join(ROOT, "include", "kvq.h")) as f:
        src = f.read()
    return set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq?_\w+)\s*\(", src))


def test_library_exports_every_declared_symbol(kb):
    declared = declared_symbols()
    assert len(declared) == 27
    for name in declared:
        assert hasattr(kb.LIB, name), name
    assert declared == set(kb.EXPORTS)
    assert kb.kvq_version().startswith("kvq ")


def formats():
    for bits in (8, 4, 2):
        for axis in (0, 1):
            for g in (0, 1, 8, 32, 64, 100):
                for R in (0, 5, 1000):
                    yield ("sym", bits, axis, g, R, O.F32, O.NONE)
                    yield ("sym", bits, axis, g, R, O.BF16, O.NONE)
                    yield ("asym", bits, axis, g, R, O.BF16, O.BF16)
                    yield ("asym", bits, axis, g, R, O.F32, O.I8)


def test_sizes_match_oracle(kb):
    for (mode, bits, axis, g, R, sd, zd) in formats():
        for shape in ((3, 77, 16), (1, 256, 128), (2, 0, 8), (0, 5, 8), (4, 9, 24)):
            for xd in (O.F32, O.BF16):
                if mode == "sym":
                    oq = O.QParams.sym(bits, axis=axis, group=g, residual=R, scale_dtype=sd)
                    kq = kb.QParams.sym(bits, axis=axis, group=g, residual=R, scale_dtype=sd)
                else:
                    qmin, qmax = (0, (1 << bits) - 1) if bits < 8 else (-128, 127)
                    oq = O.QParams.asym(bits, qmin, qmax, axis=axis, group=g, residual=R, scale_dtype=sd, zero_dtype=zd)
                    kq = kb.QParams.asym(bits, qmin, qmax, axis=axis, group=g, residual=R, scale_dtype=sd, zero_dtype=zd)
                got = kb.kvq_quantized_sizes(shape, xd, kq)
                assert got[:4] == O.sizes(shape, xd, oq), (shape, xd, kq)


def test_compression_ratios_match_oracle(kb):
    rng = np.random.default_rng(0)
    for _ in range(100):
        v = [int(a) for a in rng.integers(1, 1 << 40, 5)]
        assert kb.kvq_compression_ratio(*v) == O.compression_ratio(*v)
    assert kb.kvq_compression_ratio(10, 0, 0, 0, 0) == 0.0
    assert kb.kvq_token_compression_ratio(131072, 2048) == 64.0
    for bad in ((10, 0), (10, 11), (0, 0), (-3, 1)):
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_token_compression_ratio(*bad)
        assert e.value.status == kb.EINVAL


def test_bad_formats_rejected(kb):
    bad = [kb.QParams(3, kb.SYM, -3, 3),
           kb.QParams.sym(4, qmax=8),
           kb.QParams.sym(4, qmax=0),
           kb.QParams.asym(4, 5, 5),
           kb.QParams.asym(4, 0, 16),
           kb.QParams.asym(4, -9, 7),
           kb.QParams(4, kb.SYM, -7, 7, zero_dtype=kb.I8),
           kb.QParams.asym(4, 0, 15, zero_dtype=kb.NONE),
           kb.QParams.sym(4, scale_dtype=kb.I8),
           kb.QParams(4, 7, 0, 7),
           kb.QParams(4, kb.SYM, -7, 7, axis=5),
           kb.QParams.sym(4, group=-1),
           kb.QParams.sym(4, residual=-2)]
    for qp in bad:
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_quantized_sizes((1, 4, 8), kb.F32, qp)
        assert e.value.status == kb.EINVAL, qp
    for shape in ((1, 4, 3), (-1, 4, 8), (1 << 30, 1 << 30, 8)):
        with pytest.raises(kb.KvqError):
            kb.kvq_quantized_sizes(shape, kb.F32, kb.QParams.sym(4))
    with pytest.raises(kb.KvqError):
        kb.kvq_quantized_sizes((1, 4, 8), kb.I8, kb.QParams.sym(4))


def test_calls_rejected_before_launch(kb):
    """Every rejected call returns before touching the device: NULL buffers,
    short workspaces, empty statistics, bad selection arguments."""
    qp = kb.QParams.sym(4, axis=kb.ALONG_C, group=32)
    shape = (2, 16, 64)
    fake = 1 << 20  # never dereferenced: validation fails first
    with pytest.raises(kb.KvqError) as e:
        kb.kvq_quantize(None, kb.BF16, shape, qp, fake, fake, None, None, None, 0, 0)
    assert e.value.status == kb.EINVAL and "x" in str(e.value)
    with pytest.raises(kb.KvqError):
        kb.kvq_quantize(fake, kb.BF16, shape, qp, None, fake, None, None, None, 0, 0)
    with pytest.raises(kb.KvqError):       # residual window without a residual buffer
        kb.kvq_quantize(fake, kb.BF16, shape, kb.QParams.sym(4, residual=4), fake, fake, None, None, None, 0, 0)
    with pytest.raises(kb.KvqError):       # asymmetric without a zero buffer
        kb.kvq_quantize(fake, kb.BF16, shape, kb.QParams.asym(4, 0, 15, zero_dtype=kb.BF16), fake, fake, None,
                        None, None, 0, 0)
    with pytest.raises(kb.KvqError) as e:  # long groups need the workspace
        kb.kvq_quantize(fake * 16, kb.BF16, (1, 1024, 64), kb.QParams.sym(8, group=0), fake * 16, fake * 16,
                        None, None, None, 0, 0)
    assert e.value.status == kb.EWORKSPACE
    with pytest.raises(kb.KvqError) as e:
        kb.kvq_error_stats(fake, kb.BF16, fake, fake, None, None, (0, 16, 64), qp, fake, fake, 1 << 20, 0)
    assert e.value.status == kb.EINVAL
    with pytest.raises(kb.KvqError) as e:
        kb.kvq_error_stats(fake, kb.BF16, fake, fake, None, None, shape, qp, fake, None, 0, 0)
    assert e.value.status == kb.EWORKSPACE
    with pytest.raises(kb.KvqError):
        kb.kvq_dequantize(fake, fake, None, None, shape, qp, None, kb.BF16, 0)
    with pytest.raises(kb.KvqError):
        kb.kvq_dequantize(fake, fake, None, None, shape, qp, fake, kb.I8, 0)

    ws = kb.kv_select_workspace(4, 100)
    assert ws > 4 * 100 * 4
    sel = dict(hist=fake, heads=4, steps=8, T=100, keep=fake, scores=None, workspace=fake, workspace_B=ws)
    for budget, window in ((0, 0), (5, 6), (5, -1)):
        with pytest.raises(kb.KvqError) as e:
            kb.kv_h2o_select(budget=budget, window=window, stream=0, **sel)
        assert e.value.status == kb.EINVAL
    with pytest.raises(kb.KvqError):
        kb.kv_h2o_select(fake, 4, 0, 100, 10, 2, fake, None, fake, ws, 0)          # steps < 1
    for obs in (0, 9):
        with pytest.raises(kb.KvqError):
            kb.kv_snapkv_select(fake, 4, 8, 100, obs, 10, 2, fake, None, fake, ws, 0)
    with pytest.raises(kb.KvqError) as e:
        kb.kv_h2o_select(fake, 4, 8, 100, 10, 2, fake, None, fake, ws - 1, 0)
    assert e.value.status == kb.EWORKSPACE
    with pytest.raises(kb.KvqError):
        kb.kv_h2o_select(None, 4, 8, 100, 10, 2, fake, None, fake, ws, 0)
    with pytest.raises(kb.KvqError):
        kb.kv_select_workspace(1, 1 << 32)
    # compaction: K outside [0, T], bad dtype, NULL buffers
    for K in (-1, 101):
        with pytest.raises(kb.KvqError):
            kb.kv_compact(fake, kb.BF16, 4, 100, 128, fake, K, fake, 0)
    with pytest.raises(kb.KvqError):
        kb.kv_compact(fake, kb.NONE, 4, 100, 128, fake, 10, fake, 0)
    with pytest.raises(kb.KvqError):
        kb.kv_compact(fake, kb.BF16, 4, 100, 128, None, 10, fake, 0)
    assert "NULL" in kb.kvq_last_error()
    # the K+V form checks both tensors and both outputs
    for K in (-1, 101):
        with pytest.raises(kb.KvqError):
            kb.kv_compact_kv(fake, fake, kb.BF16, 4, 100, 128, fake, K, fake, fake, 0)
    for args in ((None, fake, fake, fake), (fake, None, fake, fake), (fake, fake, None, fake), (fake, fake, fake, None)):
        k, v, ok, ov = args
        with pytest.raises(kb.KvqError):
            kb.kv_compact_kv(k, v, kb.BF16, 4, 100, 128, fake, 10, ok, ov, 0)
        assert "NULL" in kb.kvq_last_error()
    with pytest.raises(kb.KvqError):
        kb.kv_compact_kv(fake, fake, kb.F32, 4, 100, 128, fake + 2, 10, fake, fake, 0)


def test_misaligned_buffers_rejected(kb):
    """Typed buffers must be aligned to their element size and workspaces to
    16 bytes; otherwise the call is rejected on the host."""
    base = 1 << 24
    qp = kb.QParams.sym(8, axis=kb.ALONG_T, group=16)            # float32 scale
    shape = (1, 32, 16)
    with pytest.raises(kb.KvqError) as e:
        kb.kvq_quantize(base, kb.F32, shape, qp, base, base + 2, None, None, None, 0, 0)
    assert e.value.status == kb.EINVAL and "aligned" in str(e.value)
    with pytest.raises(kb.KvqError):
        kb.kvq_quantize(base + 2, kb.F32, shape, qp, base, base, None, None, None, 0, 0)
    with pytest.raises(kb.KvqError):
        kb.kvq_dequantize(base, base, None, None, shape, qp, base + 1, kb.BF16, 0)
    with pytest.raises(kb.KvqError):
        kb.kvq_error_stats(base, kb.F32, base, base, None, None, shape, qp, base + 4, base, 1 << 20, 0)
    ws = kb.kv_select_workspace(2, 64)
    with pytest.raises(kb.KvqError):
        kb.kv_h2o_select(base + 2, 2, 4, 64, 8, 2, base, None, base, ws, 0)
    with pytest.raises(kb.KvqError):
        kb.kv_h2o_select(base, 2, 4, 64, 8, 2, base, None, base + 8, ws, 0)
    with pytest.raises(kb.KvqError):
        kb.kv_compact(base, kb.BF16, 2, 64, 8, base + 1, 4, base, 0)


def test_wait_timeouts_rejects_null(kb):
    """Argument checks run before the device synchronisation: no GPU needed."""
    assert kb.LIB.kvq_wait_timeouts(None) == kb.EINVAL
    assert "count" in kb.LIB.kvq_last_error().decode()


def test_attend_rejected_before_launch(kb):
    """Fused decode attention: shape, group, format and buffer checks on the host."""
    fake = 1 << 20  # never dereferenced: validation fails first
    kq = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_T, group=64, residual=128, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    vq = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_C, group=64, residual=128, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    shape = (2, 1000, 128)
    wB = kb.kvq_attend_workspace(shape, 2)
    assert wB == 2 * 2 * 4 * (2 + 128) * 4           # outer x group x ceil(T/256) splits x (max, sum, C) floats
    args = [fake] * 4

    def call(q=fake, group=2, k=None, v=None, kp=kq, vp=vq, sh=shape, out=fake, ws=fake, wsB=wB):
        kb.kvq_attend_decode(q, group, *(k or args), kp, *(v or args), vp, sh, out, ws, wsB, 0)

    cases = [
        (dict(q=None), kb.EINVAL),
        (dict(out=None), kb.EINVAL),
        (dict(group=0), kb.EINVAL),
        (dict(sh=(2, 0, 128)), kb.EINVAL),
        (dict(vp=kb.QParams.asym(4, 0, 15, axis=kb.ALONG_C, group=64, residual=5, scale_dtype=kb.BF16,
                                 zero_dtype=kb.BF16)), kb.EINVAL),
        (dict(k=[fake + 4, fake, fake, fake]), kb.EINVAL),               # codes not 16-byte aligned
        (dict(sh=(2, 1000, 64)), kb.EUNSUPPORTED),
        (dict(group=3), kb.EUNSUPPORTED),
        (dict(kp=vq), kb.EUNSUPPORTED),                                  # K grouped per token
        (dict(vp=kb.QParams.asym(8, 0, 255, axis=kb.ALONG_C, group=64, residual=128, scale_dtype=kb.BF16,
                                 zero_dtype=kb.BF16)), kb.EUNSUPPORTED),  # bit widths differ
        (dict(kp=kb.QParams.asym(4, 0, 15, axis=kb.ALONG_T, group=48, residual=128, scale_dtype=kb.BF16,
                                 zero_dtype=kb.BF16)), kb.EUNSUPPORTED),  # K groups not a multiple of 32
        (dict(ws=None), kb.EWORKSPACE),
        (dict(wsB=wB - 1), kb.EWORKSPACE),
    ]
    for kw, status in cases:
        with pytest.raises(kb.KvqError) as e:
            call(**kw)
        assert e.value.status == status, (kw, str(e.value))


def test_rotate_rejected_before_launch(kb):
    fake = 1 << 20  # never dereferenced: validation fails first
    for shape, xd, od, signs, x, status in (
            ((2, 10, 48), kb.BF16, kb.BF16, fake, fake, kb.EUNSUPPORTED),     # C not a power of two
            ((2, 10, 16), kb.BF16, kb.BF16, fake, fake, kb.EUNSUPPORTED),     # C below 32
            ((2, 10, 2048), kb.F32, kb.F32, fake, fake, kb.EUNSUPPORTED),     # C above 1024
            ((2, 10, 128), kb.I8, kb.BF16, fake, fake, kb.EINVAL),            # source dtype
            ((2, 10, 128), kb.BF16, kb.I8, fake, fake, kb.EINVAL),            # output dtype
            ((2, 10, 128), kb.BF16, kb.BF16, None, fake, kb.EINVAL),          # no signs
            ((2, 10, 128), kb.BF16, kb.BF16, fake, None, kb.EINVAL),          # no input
            ((2, 10, 128), kb.BF16, kb.BF16, fake, fake + 4, kb.EINVAL)):     # misaligned
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_rotate(x, xd, shape, signs, False, fake, od, 0)
        assert e.value.status == status, (shape, str(e.value))
    kb.kvq_rotate(None, kb.BF16, (0, 10, 128), None, False, None, kb.BF16, 0)   # empty: nothing to do


def test_fused_rotation_rejected_before_launch(kb):
    """kvq_rotate_quantize / kvq_dequantize_rotate: formats and shapes the
    fused kernels do not take, missing or misaligned buffers."""
    fake = 1 << 20  # never dereferenced: validation fails first
    v64 = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_C, group=64, residual=4, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    cases = (
        ((2, 10, 128), kb.F32, v64, fake, fake, kb.EUNSUPPORTED),                                   # fp32 tensor
        ((2, 10, 128), kb.BF16, kb.QParams.sym(4, axis=kb.ALONG_T, group=64), fake, fake, kb.EUNSUPPORTED),  # along T
        ((2, 10, 128), kb.BF16, kb.QParams.sym(4, axis=kb.ALONG_C, group=16), fake, fake, kb.EUNSUPPORTED),  # g < 32
        ((2, 10, 128), kb.BF16, kb.QParams.sym(4, axis=kb.ALONG_C, group=96), fake, fake, kb.EUNSUPPORTED),  # g not 2^k
        ((2, 10, 512), kb.BF16, v64, fake, fake, kb.EUNSUPPORTED),                                  # C > 256
        ((2, 10, 48), kb.BF16, kb.QParams.sym(4, axis=kb.ALONG_C, group=0), fake, fake, kb.EUNSUPPORTED),  # C
        ((2, 10, 128), kb.BF16, v64, None, fake, kb.EINVAL),                                        # no signs
        ((2, 10, 128), kb.BF16, v64, fake, None, kb.EINVAL),                                        # no tensor
        ((2, 10, 128), kb.BF16, v64, fake, fake + 8, kb.EINVAL),                                    # misaligned
        ((2, 10, 128), kb.BF16, kb.QParams.sym(4, qmax=9, axis=kb.ALONG_C, group=64), fake, fake, kb.EINVAL),  # format
    )
    for shape, dt, qp, signs, x, status in cases:
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_rotate_quantize(x, dt, shape, signs, qp, fake, fake, fake, fake, 0)
        assert e.value.status == status, ("quantize", shape, str(e.value))
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_dequantize_rotate(fake, fake, fake, fake, shape, qp, signs, x, dt, 0)
        assert e.value.status == status, ("dequantize", shape, str(e.value))
    # codes misaligned
    with pytest.raises(kb.KvqError) as e:
        kb.kvq_rotate_quantize(fake, kb.BF16, (2, 10, 128), fake, v64, fake + 4, fake, fake, fake, 0)
    assert e.value.status == kb.EINVAL
    # empty tensors: nothing to do
    kb.kvq_rotate_quantize(None, kb.BF16, (0, 10, 128), None, v64, None, None, None, None, 0)
    kb.kvq_dequantize_rotate(None, None, None, None, (3, 0, 128), v64, None, None, kb.BF16, 0)


def test_append_rejected_before_launch(kb):
    """Streaming append: bad counters, block/group mismatch, a store too small
    for the flushes, missing workspace -- rejected with the counters unchanged."""
    fake = 1 << 20  # never dereferenced: validation fails first
    qp = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_T, group=32, residual=16, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    shape = (2, 64, 128)                                   # store of 64 tokens
    wB = kb.kvq_append_workspace(shape, kb.BF16, qp, 32)
    assert wB > 0
    with pytest.raises(kb.KvqError) as e:
        kb.kvq_append_workspace(shape, kb.BF16, qp, 48)   # block not a multiple of the group
    assert e.value.status == kb.EINVAL
    args = dict(codes=fake, scale=fake, zero=fake, resid=fake, ws=fake, wsB=wB)

    def call(n=1, tq=0, nres=0, **kw):
        a = dict(args, **kw)
        return kb.kvq_append(fake, n, kb.BF16, shape, qp, 32, a["codes"], a["scale"], a["zero"], a["resid"], tq,
                             nres, a["ws"], a["wsB"], 0)

    for kw, status in ((dict(tq=5), kb.EINVAL), (dict(nres=48), kb.EINVAL), (dict(n=-1), kb.EINVAL),
                       (dict(n=120), kb.EINVAL),             # 3 flushes of 32 need 96 > 64 store tokens
                       (dict(n=50, resid=None), kb.EINVAL),  # 50 tokens fill the 48-row buffer once
                       (dict(n=50, ws=None), kb.EWORKSPACE), (dict(n=50, wsB=wB - 1), kb.EWORKSPACE)):
        with pytest.raises(kb.KvqError) as e:
            call(**kw)
        assert e.value.status == status, (kw, str(e.value))


def test_append_kv_rejected_before_launch(kb):
    """kvq_append_kv: residual windows that differ, bad counters, a store too
    small, a missing workspace -- rejected, counters unchanged."""
    import ctypes
    fake = 1 << 20
    shape = (2, 256, 128)
    kq = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_T, group=64, residual=128, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    vq = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_C, group=64, residual=128, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    v_other = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_C, group=64, residual=64, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    wB = kb.kvq_append_kv_workspace(shape, kb.BF16, kq, vq, 64)
    assert wB == kb.kvq_append_workspace(shape, kb.BF16, kq, 64) + kb.kvq_append_workspace(shape, kb.BF16, vq, 64)
    bufs = (fake, fake, fake, fake)
    for kw, status in (
            (dict(vqp=v_other), kb.EINVAL),                          # residual windows differ
            (dict(tq=3), kb.EINVAL),                                 # tq not a multiple of block
            (dict(nres=192), kb.EINVAL),                             # nres = residual + block
            (dict(n=-1), kb.EINVAL),
            (dict(tq=256, nres=191, n=1), kb.EINVAL),                # the flush does not fit the store
            (dict(nres=191, n=1, ws=None, wsB=0), kb.EWORKSPACE),    # a flush without workspace
            (dict(nres=191, n=1, wsB=wB - 1), kb.EWORKSPACE),
            (dict(k_new=None), kb.EINVAL),
            (dict(v_new=fake + 1), kb.EINVAL)):                      # misaligned bf16 rows
        a = dict(k_new=fake, v_new=fake, n=1, vqp=vq, tq=0, nres=0, ws=fake, wsB=wB)
        a.update(kw)
        t, r = ctypes.c_int64(a["tq"]), ctypes.c_int64(a["nres"])
        with pytest.raises(kb.KvqError) as e:
            kb._check(kb.LIB.kvq_append_kv(a["k_new"], a["v_new"], a["n"], kb.BF16, ctypes.byref(kb._shape(shape)),
                                           ctypes.byref(kq.c()), ctypes.byref(a["vqp"].c()), 64, *bufs, *bufs,
                                           ctypes.byref(t), ctypes.byref(r), a["ws"], a["wsB"], None))
        assert e.value.status == status, (kw, str(e.value))
        assert (t.value, r.value) == (a["tq"], a["nres"]), kw


def test_kv_appender_reports_errors_and_keeps_counters(kb):
    """KVAppender: a rejected call raises KvqError and leaves tq / nres as they were."""
    fake = 1 << 20

    class FakeTensor:                           # only data_ptr() and numel() are used
        def __init__(self, p, n=0):
            self.p, self.n = p, n

        def data_ptr(self):
            return self.p

        def numel(self):
            return self.n

    shape = (2, 256, 128)
    kq = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_T, group=64, residual=128, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    vq = kb.QParams.asym(4, 0, 15, axis=kb.ALONG_C, group=64, residual=128, scale_dtype=kb.BF16, zero_dtype=kb.BF16)
    bufs = tuple(FakeTensor(fake) for _ in range(4))
    ws = FakeTensor(fake, kb.kvq_append_kv_workspace(shape, kb.BF16, kq, vq, 64))
    app = kb.KVAppender(shape, kb.BF16, kq, vq, 64, bufs, bufs, ws, tq=0, nres=191, stream=0)
    with pytest.raises(kb.KvqError) as e:
        app.append(FakeTensor(fake + 1), FakeTensor(fake), 1)      # misaligned rows: rejected before launch
    assert e.value.status == kb.EINVAL
    assert (app.tq, app.nres) == (0, 191)
    app.set_counters(3, 0)
    with pytest.raises(kb.KvqError) as e:
        app.append(FakeTensor(fake), FakeTensor(fake), 1)          # tq not a multiple of block
    assert e.value.status == kb.EINVAL and (app.tq, app.nres) == (3, 0)


def test_mixed_rejected_before_launch(kb):
    fake = 1 << 20
    assert kb.kvq_mixed_sizes((2, 10, 128)) == (2 * 10 * 128 * 2, 2 * 11 * 8, 2 * 3)
    for shape, x, off, status in (((2, 10, 96), fake, fake, kb.EUNSUPPORTED), ((2, 10, 128), None, fake, kb.EINVAL),
                                  ((2, 10, 128), fake + 1, fake, kb.EINVAL), ((2, 10, 128), fake, fake + 4, kb.EINVAL),
                                  ((2, 10, 128), fake + 2, fake, kb.EINVAL)):     # rows read 16 bytes at a time
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_mixed_quantize(x, fake, shape, fake, off, fake, 0)
        assert e.value.status == status, (shape, str(e.value))
    for shape, x, off, status in (((2, 10, 128), fake, fake, kb.EINVAL),):       # stream_buf by bulk copies
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_mixed_quantize(x, fake, shape, fake + 2, off, fake, 0)
        assert e.value.status == status, (shape, str(e.value))
    for sbuf, out in ((fake, None), (fake, fake + 2), (fake + 2, fake)):
        with pytest.raises(kb.KvqError) as e:
            kb.kvq_mixed_dequantize(sbuf, fake, fake, (2, 10, 128), out, 0)
        assert e.value.status == kb.EINVAL

