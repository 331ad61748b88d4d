"""CUDA per-token mixed precision vs the CPU oracle.

Every token's record must equal the oracle's quantization of that token alone
in its tag's format ("大模型KV缓存自适应量化实战" §3.1: 2 and 4 bits symmetric,
8 bits asymmetric [0, 255], 16 bits as is; per token, bf16 scale and zero
point), laid out as include/kvq.h describes (records in token order, offsets
by prefix sums, 2-bit tags); everything bit for bit, the dequantized values
too.
"""
import zlib

import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def formats(C):
    return [O.QParams.sym(2, axis=O.ALONG_C, group=C, scale_dtype=O.BF16),
            O.QParams.sym(4, axis=O.ALONG_C, group=C, scale_dtype=O.BF16),
            O.QParams.asym(8, 0, 255, axis=O.ALONG_C, group=C, scale_dtype=O.BF16, zero_dtype=O.BF16)]


def expected(X, tags):
    """(stream per slice, offsets, packed tags, dequantized) from the oracle."""
    outer, T, C = X.shape
    F = formats(C)
    streams, offs, deq = [], np.zeros((outer, T + 1), np.int64), np.zeros_like(X)
    for o in range(outer):
        recs = []
        for t in range(T):
            g = int(tags[o, t]) & 3
            row = X[o, t].reshape(1, 1, C)
            if g == 3:
                recs.append(row.tobytes())
                deq[o, t] = X[o, t]
            else:
                q = O.quantize(row, O.BF16, F[g])
                recs.append(q.codes.tobytes() + q.scale.tobytes() + q.zero.tobytes())
                deq[o, t] = O.dequantize(q, (1, 1, C), F[g], O.BF16)[0, 0]
            offs[o, t + 1] = offs[o, t] + len(recs[-1])
        streams.append(b"".join(recs))
    t2 = np.zeros((outer, (T + 3) // 4), np.uint8)
    for t in range(T):
        t2[:, t // 4] |= ((tags[:, t] & 3) << (2 * (t % 4))).astype(np.uint8)
    return streams, offs, t2, deq


def expected_one_level(X, tag):
    """expected() for a cache whose tokens all carry one tag below 3, from whole-
    tensor oracle calls: per-token groups give one record per token row."""
    outer, T, C = X.shape
    qp = formats(C)[tag]
    q = O.quantize(X, O.BF16, qp)
    parts = [q.codes.reshape(outer, T, -1), q.scale.view(np.uint8).reshape(outer, T, -1)]
    if q.zero.size:
        parts.append(q.zero.view(np.uint8).reshape(outer, T, -1))
    recs = np.concatenate(parts, axis=2)
    rb = recs.shape[2]
    offs = np.tile(np.arange(T + 1, dtype=np.int64) * rb, (outer, 1))
    streams = [recs[o].tobytes() for o in range(outer)]
    t2 = np.zeros((outer, (T + 3) // 4), np.uint8)
    for j in range(4):
        t2[:, : (T - j + 3) // 4] |= np.uint8(tag << (2 * j))
    deq = O.dequantize(q, X.shape, qp, O.BF16).reshape(X.shape)
    return streams, offs, t2, deq


def run(b, shape, tags, kind="normal", seed=0, one_level=None):
    import torch
    outer, T, C = shape
    rng = np.random.default_rng(seed)
    if kind == "normal":
        x = W.random_kv(rng, shape)
    elif kind == "zeros":
        x = np.zeros(shape, np.float32)
    else:                                           # constant rows
        x = np.full(shape, 1.5, np.float32)
    X = W.to_bf16_bits(x)
    sB, oB, tB = b.kvq_mixed_sizes(shape)
    dev = torch.device("cuda")
    xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
    td = torch.from_numpy(np.ascontiguousarray(tags, dtype=np.uint8)).cuda()
    g = Guarded()                      # canary bytes around every written buffer
    sbuf = g.alloc(sB)
    off = g.alloc(oB).view(torch.int64)
    t2 = g.alloc(tB)
    out = g.alloc(outer * T * C * 2).view(torch.bfloat16).view(shape)
    b.kvq_mixed_quantize(xd, td, shape, sbuf, off, t2)
    g.check("kvq_mixed_quantize")
    b.kvq_mixed_dequantize(sbuf, off, t2, shape, out)
    g.check("kvq_mixed_dequantize")
    streams, offs, t2w, deq = expected(X, tags) if one_level is None else expected_one_level(X, one_level)
    got_off = off.cpu().numpy().reshape(outer, T + 1)
    assert np.array_equal(got_off, offs), "record offsets differ"
    assert np.array_equal(t2.cpu().numpy().reshape(outer, -1), t2w), "packed tags differ"
    sb = sbuf.cpu().numpy().reshape(outer, T * 2 * C)
    for o in range(outer):
        assert sb[o, : offs[o, T]].tobytes() == streams[o], f"records of slice {o} differ"
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), deq), "dequantized values differ"


@pytest.mark.parametrize("C", [64, 128, 256])
def test_mixed_random_tags(b, C):
    rng = np.random.default_rng(C)
    shape = (2, 301, C)
    run(b, shape, rng.integers(0, 4, shape[:2]), seed=zlib.crc32(repr(C).encode()))


def test_mixed_random_tags_long_slices(b):
    """Thousands of tokens per slice at C = 64: 20 sub-rounds of 256 tokens,
    one per CTA, the last one ragged (5003 = 19 * 256 + 139); every CTA but the
    first sums the record bytes of the tokens before it."""
    rng = np.random.default_rng(5003)
    shape = (2, 5003, 64)
    run(b, shape, rng.integers(0, 4, shape[:2]), seed=11)


@pytest.mark.parametrize("tag", [0, 1, 2])
def test_mixed_one_level_beyond_one_grid_pass(b, tag):
    """200003 tokens in one slice: 32 CTAs of 49 sub-rounds of 128 tokens
    each, the last one ragged; record offsets beyond 2^24 bytes."""
    T = 200003
    shape = (1, T, 128)
    run(b, shape, np.full(shape[:2], tag), seed=tag + 20, one_level=tag)


@pytest.mark.parametrize("tag", [0, 1, 2, 3])
def test_mixed_single_level(b, tag):
    shape = (3, 70, 128)
    run(b, shape, np.full(shape[:2], tag), seed=tag)


@pytest.mark.parametrize("kind", ["zeros", "const"])
def test_mixed_degenerate_rows(b, kind):
    shape = (1, 40, 128)
    run(b, shape, np.arange(40).reshape(1, 40) % 4, kind=kind)


def test_mixed_memory_matches_the_tag_mix(b):
    """The bytes a slice uses follow from its tags alone: a quarter of each
    level at C = 128 averages (34 + 66 + 132 + 256) / 4 = 122 bytes per token."""
    shape = (1, 400, 128)
    tags = np.tile(np.arange(4), 100).reshape(1, 400)
    _, offs, _, _ = expected(W.to_bf16_bits(np.ones(shape, np.float32)), tags)
    assert offs[0, -1] == 100 * (34 + 66 + 132 + 256)
    run(b, shape, tags, seed=3)
