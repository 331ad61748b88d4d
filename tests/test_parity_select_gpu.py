"""CUDA H2O / SnapKV selection and compaction vs the CPU oracle.

Scores must be bit-exact (same float32 adds in the same step order, same
division); keep indices bit-exact; compacted rows bit-exact.
"""
import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb, to_host
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def gpu_select(b, hist, budget, window, obs=None, offset=0, want_scores=True):
    """One selection call; keep, scores and the workspace are guarded
    windows whose surrounding canary bytes must survive the call."""
    import torch
    H, S, T = hist.shape
    raw = torch.zeros(hist.size + 16, dtype=torch.float32, device="cuda")
    h = raw[offset:offset + hist.size]
    h.copy_(torch.from_numpy(hist.ravel()).cuda())
    g = Guarded()
    K = min(budget, T)
    keep_w = g.alloc(H * K * 4)
    keep = keep_w.view(torch.int32).view(H, K) if keep_w is not None else torch.empty((H, K), dtype=torch.int32,
                                                                                        device="cuda")
    scores = None
    if want_scores:
        sw = g.alloc(H * T * 4)
        scores = sw.view(torch.float32).view(H, T) if sw is not None else torch.empty((H, T), device="cuda")
    wB = b.kv_select_workspace(H, T)
    ws = g.alloc(wB)
    if obs is None:
        b.kv_h2o_select(h, H, S, T, budget, window, keep, scores, ws, wB)
    else:
        b.kv_snapkv_select(h, H, S, T, obs, budget, window, keep, scores, ws, wB)
    torch.cuda.synchronize()
    g.check("selection")
    return to_host(keep), (to_host(scores) if want_scores else None)


def compare(b, hist, budget, window, obs=None, offset=0):
    if obs is None:
        ok, osc = O.h2o_select(hist, budget, window)
    else:
        ok, osc = O.snapkv_select(hist, obs, budget, window)
    gk, gs = gpu_select(b, hist, budget, window, obs, offset)
    assert np.array_equal(gs.view(np.uint32), osc.view(np.uint32)), "scores differ"
    assert np.array_equal(gk, ok), "keep sets differ"
    # without the optional scores output the keep set is unchanged
    gk2, _ = gpu_select(b, hist, budget, window, obs, offset, want_scores=False)
    assert np.array_equal(gk2, ok)


@pytest.mark.parametrize("T", [1, 3, 5, 100, 1023, 1024, 1025, 4096, 5000, 20000])
def test_h2o_random(b, T):
    rng = np.random.default_rng(T)
    hist = W.random_history(rng, 3, 7, T, planted=min(8, T))
    for budget, window in ((1, 0), (1, 1), (min(64, T), 16 if T > 16 else 0), (T, 3), (T + 5, 2),
                           (max(1, T // 2), min(T // 4, 128)), (300, 300), (2 * T + 1, 0)):
        if window > budget:
            continue
        compare(b, hist, budget, window)


@pytest.mark.parametrize("T", [7, 256, 3000])
def test_snapkv_random(b, T):
    rng = np.random.default_rng(T + 1)
    hist = W.random_history(rng, 2, 12, T)
    for obs in (1, 4, 12, 5):
        compare(b, hist, min(T, 40), min(T, 10) // 2, obs=obs)


def test_ties_signed_zeros_and_flat_rows(b):
    """Equal scores are broken by the lowest index; -0 and +0 tie."""
    rng = np.random.default_rng(1)
    T = 3000
    hist = np.zeros((4, 3, T), np.float32)
    hist[0] = rng.integers(0, 4, (3, T)) / 4.0                 # heavy ties
    hist[1] = 1.0 / T                                            # flat rows: every score equal
    hist[2] = rng.choice(np.array([0.0, -0.0], np.float32), (3, T))
    hist[3] = rng.integers(0, 2, (3, T)).astype(np.float32)
    hist[3, :, ::7] = -0.0
    for budget, window in ((100, 10), (1500, 0), (2999, 1), (7, 7), (1, 0)):
        compare(b, hist, budget, window)
        compare(b, hist, budget, window, obs=2)


# Context lengths above 2^19 tokens take the other selection algorithm: a
# level-1 histogram in the column sums, then three radix digits (12, 12 and 8
# key bits) each by a histogram pass over the scores and a per-head digit
# pick, per-chunk counts of keys above / equal to the k-th key, and an emit
# pass that writes the heavy hitters (ties in index order) and the window.
LONG_T = [524289, 600000]


@pytest.mark.parametrize("T", LONG_T)
def test_h2o_long_context_radix_path(b, T):
    rng = np.random.default_rng(T)
    hist = W.random_history(rng, 2, 4, T, planted=64, window=128)
    for budget, window in ((1, 0), (2048, 128), (2048, 0), (T - 1, 128), (T - 1, 0), (T, 128), (5000, 5000)):
        compare(b, hist, budget, window)


@pytest.mark.parametrize("T", LONG_T)
def test_snapkv_long_context_radix_path(b, T):
    rng = np.random.default_rng(T + 3)
    hist = W.random_history(rng, 2, 4, T, planted=64)
    for budget, window in ((2048, 128), (1, 0)):
        compare(b, hist, budget, window, obs=2)


def test_long_context_flat_and_tied_heads(b):
    """Every score of head 0 tied (flat rows): all three digit levels resolve
    to one key and the tie pass keeps the lowest indices.  Head 1: a few
    score values only, so the k-th key has many ties; head 2: signed zeros."""
    rng = np.random.default_rng(7)
    T = 600000
    hist = np.empty((3, 2, T), np.float32)
    hist[0] = 1.0 / T
    hist[1] = rng.integers(0, 5, (2, T)) / 8.0
    hist[2] = rng.choice(np.array([0.0, -0.0, 2.0 ** -20], np.float32), (2, T), p=[0.45, 0.45, 0.1])
    for budget, window in ((2048, 128), (1, 0), (300000, 17), (T - 1, 1)):
        compare(b, hist, budget, window)
    compare(b, hist, 2048, 128, obs=1)


def test_long_context_unaligned_history(b):
    """T > 2^19 with a history that is not 16-byte aligned and T not a
    multiple of 4: the scalar column-sum kernel of the radix path."""
    rng = np.random.default_rng(11)
    T = 524291
    hist = W.random_history(rng, 2, 3, T, planted=16)
    compare(b, hist, 2048, 128, offset=1)
    compare(b, hist, 777, 0, offset=3, obs=2)


def test_unaligned_history_scalar_path(b):
    rng = np.random.default_rng(2)
    hist = W.random_history(rng, 2, 5, 1000)
    compare(b, hist, 50, 8, offset=1)
    compare(b, hist, 50, 8, offset=3, obs=3)


def test_tiny_config_selection(b):
    """Tiny workload: history [32 steps, 256 tokens], B=64, W=16, H2O and
    SnapKV on the row mean (obs_window = all 32 steps)."""
    _, hist = W.tiny_inputs(0)
    compare(b, hist, 64, 16)
    compare(b, hist, 64, 16, obs=32)
    keep, _ = O.h2o_select(hist, 64, 16)
    assert keep.shape == (1, 64) and set(range(240, 256)) <= set(keep[0].tolist())


def test_empty_inputs(b):
    hist = np.zeros((2, 3, 0), np.float32)
    gk, _ = gpu_select(b, hist, 5, 2, want_scores=False)
    assert gk.shape == (2, 0)
    gk, _ = gpu_select(b, np.zeros((0, 3, 10), np.float32), 5, 2, want_scores=False)
    assert gk.shape == (0, 5)


# ---------------------------------------------------------------- compaction


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("i8", 40), ("bf16", 3), ("f32", 1)])
def test_compact(b, dtype, D):
    import torch
    rng = np.random.default_rng(D)
    H, T, K = 3, 500, 77
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "i8": torch.int8}[dtype]
    kv = torch.from_numpy(rng.standard_normal((H, T, D)).astype(np.float32) * 10).to(tdt).cuda()
    keep = np.sort(rng.choice(T, (H, K)), axis=1).astype(np.int32)
    keep[1] = rng.permutation(T)[:K]                            # order is the caller's
    g = Guarded()
    es = kv.element_size()
    out = g.alloc(H * K * D * es).view(tdt).view(H, K, D)
    b.compact(kv, torch.from_numpy(keep).cuda(), out=out)
    g.check("kv_compact")
    host = to_host(kv)
    want = O.compact(host, keep)
    assert np.array_equal(to_host(out), want)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 32), ("f32", 16), ("f32", 256), ("bf16", 512),
                                     ("i8", 40), ("bf16", 3)])
def test_compact_kv_pair(b, dtype, D):
    """K and V through one call: rows of 64 B .. 1 KB take the batched row
    kernel, other sizes the per-piece kernel; ragged K, a permuted keep row,
    and keep entries outside [0, T) (zero rows)."""
    import torch
    rng = np.random.default_rng(D * 3 + len(dtype))
    H, T, K = 3, 500, 77
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "i8": torch.int8}[dtype]
    k = torch.from_numpy(rng.standard_normal((H, T, D)).astype(np.float32) * 10).to(tdt).cuda()
    v = torch.from_numpy(rng.standard_normal((H, T, D)).astype(np.float32) * 10).to(tdt).cuda()
    keep = np.sort(rng.choice(T, (H, K)), axis=1).astype(np.int32)
    keep[1] = rng.permutation(T)[:K]
    keep[2, 5] = -1
    keep[2, 40] = T
    g = Guarded()
    nb = H * K * D * k.element_size()
    ok = g.alloc(nb).view(tdt).view(H, K, D)
    ov = g.alloc(nb, offset=16).view(tdt).view(H, K, D)
    b.compact_kv(k, v, torch.from_numpy(keep).cuda(), out_k=ok, out_v=ov)
    g.check("kv_compact_kv")
    for src, got in ((k, ok), (v, ov)):
        host = to_host(src)
        want = O.compact(host, np.clip(keep, 0, T - 1))
        g = to_host(got)
        bad = (keep < 0) | (keep >= T)
        want[bad] = 0
        assert np.array_equal(g, want)


def test_compact_out_of_range_rows_are_zero(b):
    import torch
    kv = torch.arange(2 * 10 * 16, dtype=torch.float32, device="cuda").view(2, 10, 16)
    keep = torch.tensor([[0, 9, 10, -1], [3, 3, 100000, 2]], dtype=torch.int32, device="cuda")
    out = b.compact(kv, keep).cpu()
    assert torch.equal(out[0, 0], kv[0, 0].cpu()) and torch.equal(out[0, 1], kv[0, 9].cpu())
    assert not out[0, 2].any() and not out[0, 3].any() and not out[1, 2].any()
    assert torch.equal(out[1, 3], kv[1, 2].cpu())


def test_h2o_then_compact_matches_oracle_pipeline(b):
    import torch
    rng = np.random.default_rng(5)
    hist = W.random_history(rng, 4, 16, 4096, planted=32, window=64)
    kv = rng.standard_normal((4, 4096, 128)).astype(np.float32)
    ok, _ = O.h2o_select(hist, 256, 64)
    keep_d, _ = b.h2o_select(torch.from_numpy(hist).cuda(), 256, 64)
    out = b.compact(torch.from_numpy(kv).cuda(), keep_d)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), O.compact(kv, ok))
