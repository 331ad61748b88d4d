"""CUDA streaming append (online quantized cache) vs the CPU oracle.

Appending the T tokens of a sequence in arbitrary chunks must leave exactly
what quantizing the whole sequence at once gives, with the residual window
T - tq: the same codes, scales and zero points for the first tq tokens and the
remaining tokens, as stored, in the buffer (bit for bit), with
tq = block * max(0, floor((T - R) / block)) ("KV cache 压缩：把历史装得更小",
§带残差区的压缩预算，逐项加起来: the recent tokens stay bf16, the older ones are
quantized in groups).
"""
import zlib

import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb, kq_of, meta_np_dtype
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


CASES = [
    # bits, (qmin, qmax) or None, axis, g, R, block, C, outer, T
    (4, (0, 15), O.ALONG_T, 32, 16, 32, 128, 3, 300),        # KIVI keys
    (4, (0, 15), O.ALONG_C, 64, 16, 32, 128, 3, 300),        # KIVI values
    (8, None, O.ALONG_T, 64, 0, 64, 64, 2, 250),             # no residual window
    (2, None, O.ALONG_C, 32, 5, 1, 64, 2, 100),              # one token per flush
    (8, (-128, 127), O.ALONG_T, 16, 40, 48, 256, 1, 500),    # three groups per flush
    (4, (0, 15), O.ALONG_T, 64, 128, 64, 128, 2, 150),       # shorter than R + block: nothing flushed
]


def run(b, case, check_every=False):
    import torch
    bits, qr, axis, g, R, block, C, outer, T = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    X = W.to_bf16_bits(W.random_kv(rng, (outer, T, C)))
    if qr is None:
        oq = O.QParams.sym(bits, axis=axis, group=g, residual=R, scale_dtype=O.BF16 if bits < 8 else O.F32)
    else:
        oq = O.QParams.asym(bits, qr[0], qr[1], axis=axis, group=g, residual=R, scale_dtype=O.BF16,
                            zero_dtype=O.I8 if qr[0] < 0 else O.BF16)
    kq = kq_of(b, oq)
    shape = (outer, T, C)                                     # store capacity T tokens
    cB, sB, zB, _, _ = b.kvq_quantized_sizes(shape, b.BF16, b.QParams(*[getattr(kq, f) for f in (
        "bits", "mode", "qmin", "qmax", "axis", "group")], 0, kq.scale_dtype, kq.zero_dtype))
    dev = torch.device("cuda")
    g = Guarded()                      # canary bytes around every buffer the calls write
    codes = g.alloc(max(cB, 1), fill=0)
    scale = g.alloc(max(sB, 1), fill=0)
    zero = g.alloc(max(zB, 1), fill=0)
    resid = g.alloc(outer * (R + block) * C * 2, fill=0).view(torch.bfloat16)
    wB = b.kvq_append_workspace(shape, b.BF16, kq, block)
    ws = g.alloc(max(wB, 1))
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
    tq, nres, t = 0, 0, 0
    while t < T:
        n = int(min(T - t, rng.integers(1, 70)))
        chunk = Xd[:, t:t + n].contiguous()
        tq, nres = b.kvq_append(chunk, n, b.BF16, shape, kq, block, codes, scale, zero, resid, tq, nres, ws, wB)
        t += n
        g.check("kvq_append")
        if check_every:
            compare(b, X[:, :t], oq, tq, nres, codes, scale, zero, resid, R, block)
    compare(b, X, oq, tq, nres, codes, scale, zero, resid, R, block)


def compare(b, X, oq, tq, nres, codes, scale, zero, resid, R, block):
    import torch
    torch.cuda.synchronize()
    outer, T, C = X.shape
    assert tq == block * max(0, (T - R) // block) and nres == T - tq
    cap = codes.numel() // max(outer, 1)                       # bytes of one slice of the store
    Tcap = cap // (C * oq.bits // 8)
    want = O.quantize(X, O.BF16, O.QParams(oq.bits, oq.mode, oq.qmin, oq.qmax, oq.axis, oq.group, T - tq,
                                            oq.scale_dtype, oq.zero_dtype))
    rowB = C * oq.bits // 8
    got_codes = codes.cpu().numpy()[: outer * Tcap * rowB].reshape(outer, Tcap, rowB)[:, :tq]
    assert np.array_equal(got_codes.ravel(), want.codes), "codes differ"
    if tq:
        sd = meta_np_dtype(oq.scale_dtype)
        if oq.axis == O.ALONG_T:
            ng_cap = -(-Tcap // oq.group)
            got_s = scale.cpu().numpy().view(sd)[: outer * ng_cap * C].reshape(outer, ng_cap, C)[:, : tq // oq.group]
        else:
            ngc = -(-C // oq.group)
            got_s = scale.cpu().numpy().view(sd)[: outer * Tcap * ngc].reshape(outer, Tcap, ngc)[:, :tq]
        assert np.array_equal(got_s.ravel(), want.scale), "scales differ"
        if oq.mode == O.ASYM:
            zd = meta_np_dtype(oq.zero_dtype)
            if oq.axis == O.ALONG_T:
                got_z = zero.cpu().numpy().view(zd)[: outer * ng_cap * C].reshape(outer, ng_cap, C)[:, : tq // oq.group]
            else:
                got_z = zero.cpu().numpy().view(zd)[: outer * Tcap * ngc].reshape(outer, Tcap, ngc)[:, :tq]
            assert np.array_equal(got_z.ravel(), want.zero), "zero points differ"
    buf = resid.view(torch.int16).cpu().numpy().view(np.uint16).reshape(outer, R + block, C)[:, :nres]
    assert np.array_equal(buf, X[:, tq:]), "buffered tokens differ"


@pytest.mark.parametrize("case", CASES, ids=str)
def test_append_matches_whole_sequence_quantize(b, case):
    run(b, case)


def test_append_state_after_every_chunk(b):
    run(b, (4, (0, 15), O.ALONG_T, 16, 8, 16, 64, 2, 120), check_every=True)


# K and V of one layer through one kvq_append_kv call per chunk: each cache
# must end exactly as if quantized whole (and as kvq_append leaves it).
KV_CASES = [
    # K (bits, (qmin, qmax), g), V (bits, (qmin, qmax), g), R, block, C, outer, T, chunk sizes
    ((4, (0, 15), 64), (4, (0, 15), 64), 128, 64, 128, 3, 700, "decode"),      # KIVI formats, one token a step
    ((4, (0, 15), 32), (4, (0, 15), 64), 16, 32, 128, 2, 300, "random"),
    ((8, None, 16), (2, None, 32), 40, 48, 64, 2, 400, "random"),
    ((4, (0, 15), 64), (4, (0, 15), 64), 128, 64, 128, 2, 150, "random"),      # nothing flushed
]


def _formats(spec, axis, R):
    bits, qr, g = spec
    if qr is None:
        return O.QParams.sym(bits, axis=axis, group=g, residual=R, scale_dtype=O.BF16 if bits < 8 else O.F32)
    return O.QParams.asym(bits, qr[0], qr[1], axis=axis, group=g, residual=R, scale_dtype=O.BF16, zero_dtype=O.BF16)


@pytest.mark.parametrize("case", KV_CASES, ids=str)
def test_append_kv_matches_whole_sequence_quantize(b, case):
    import torch
    kspec, vspec, R, block, C, outer, T, chunks = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    X = {n: W.to_bf16_bits(W.random_kv(rng, (outer, T, C))) for n in ("K", "V")}
    oq = {"K": _formats(kspec, O.ALONG_T, R), "V": _formats(vspec, O.ALONG_C, R)}
    kq = {n: kq_of(b, oq[n]) for n in oq}
    shape = (outer, T, C)
    g = Guarded()
    bufs = {}
    for n in ("K", "V"):
        q0 = kq[n]
        cB, sB, zB, _, _ = b.kvq_quantized_sizes(shape, b.BF16, b.QParams(q0.bits, q0.mode, q0.qmin, q0.qmax, q0.axis,
                                                                          q0.group, 0, q0.scale_dtype, q0.zero_dtype))
        bufs[n] = (g.alloc(max(cB, 1), fill=0), g.alloc(max(sB, 1), fill=0), g.alloc(max(zB, 1), fill=0),
                   g.alloc(outer * (R + block) * C * 2, fill=0).view(torch.bfloat16))
    wB = b.kvq_append_kv_workspace(shape, b.BF16, kq["K"], kq["V"], block)
    ws = g.alloc(max(wB, 1))
    Xd = {n: torch.from_numpy(X[n].view(np.int16)).view(torch.bfloat16).cuda() for n in X}
    app = b.KVAppender(shape, b.BF16, kq["K"], kq["V"], block, bufs["K"], bufs["V"], ws)
    t, step = 0, 0
    tq, nres = 0, 0
    while t < T:
        n = 1 if chunks == "decode" else int(min(T - t, rng.integers(1, 70)))
        n = min(n, T - t)
        kc, vc = Xd["K"][:, t:t + n].contiguous(), Xd["V"][:, t:t + n].contiguous()
        if step % 2:      # the object and the plain call alternate on the same counters
            app = b.KVAppender(shape, b.BF16, kq["K"], kq["V"], block, bufs["K"], bufs["V"], ws, tq=tq, nres=nres)
            app.append(kc, vc, n)
            tq, nres = app.tq, app.nres
        else:
            tq, nres = b.kvq_append_kv(kc, vc, n, b.BF16, shape, kq["K"], kq["V"], block, bufs["K"], bufs["V"], tq,
                                       nres, ws, wB)
        t += n
        step += 1
    g.check("kvq_append_kv")
    for n in ("K", "V"):
        codes, scale, zero, resid = bufs[n]
        compare(b, X[n], oq[n], tq, nres, codes, scale, zero, resid, R, block)
