"""CUDA decode attention over a quantized cache (dequantization fused in) vs
the CPU oracle.

Both sides read the same quantized cache (the oracle's buffers, uploaded), so
the comparison isolates the attention kernel.  The oracle computes in binary64
("KV cache 压缩：把历史装得更小" §"K 的误差会改变权重，V 的误差会改变内容":
logit_t = q.k_t / sqrt(d), y = sum_t softmax(logits)_t v_t, the cache rows as
s * (q - zp) in full precision); the kernel computes in float32.

Tolerance, derived from the kernel's arithmetic (u = 2^-24,
gamma_n = n u / (1 - n u), worst case, no probabilistic model).

CUDA-core path (8-bit codes), float32 throughout:
 - a base-2 logit is a sum of C products q_c * k_tc, each rounded once when
   the K scale is folded into q, accumulated as two FMA chains of C/2 terms,
   added, and scaled by the rounded log2(e)/sqrt(C):
       |d l_t| <= gamma_{C/2+4} * log2(e)/sqrt(C) * sum_c |q_c k_tc|;
 - a weight p_t = 2^(l_t - max) then carries a relative error of at most
   ln2 * (2 max_t |d l_t| + u * spread) + 16 u (exp2f within 2 ulp, the
   online-softmax rescalings and the merges of warps and splits);
 - y = sum_t p_t v_t / sum_t p_t moves by at most twice that times
   max_t |v_tc|, plus the accumulation of at most 64 tokens per warp, the
   merges and the division: gamma_{72 + splits} * max_t |v_tc|.

Tensor-core path (2- and 4-bit codes, mma.sync bf16 x bf16 -> float32):
 - each float32 factor x = q_c * s_c (logits) or p_t * s_t (values) enters as
   bf16 hi + lo with |x - hi - lo| <= 2^-16 |x| (two 8-bit significands);
   the integer factors (code - zero point) are exact in bf16;
 - the products are exact in float32 and a logit accumulates 8 mma steps
   (16 products each) and a warp's value at most 4; taking 2 ulp per step,
   8 * 2^-22 = 2^-19 relative to the sum of magnitudes;
 - so |d l_t| <= 2^-15 * log2(e)/sqrt(C) * sum_c |q_c k_tc| (2^-16 + 2^-19 +
   a few u, doubled), and the value sums gain at most 2^-15 * max_t |v_tc|
   on top of the float32 terms above.
Tiles with residual tokens (and groups whose zero points bf16 cannot hold)
take the float32 path, so the larger bound covers every token.
"""
import math
import zlib

import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb, kq_of
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def gamma(n):
    return n * U / (1 - n * U)


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def upload(qt):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).ravel()).cuda() for a in
            (qt.codes, qt.scale, qt.zero, qt.resid)]


def bound(q, K, V, splits, tc=False):
    """Per-output tolerance (see the module docstring). q [O, G, C], K / V [O, T, C];
    tc: the tensor-core path (2- and 4-bit codes)."""
    C = q.shape[-1]
    S = np.einsum("ojc,otc->ojt", np.abs(q), np.abs(K))                 # sum_c |q_c k_tc|
    coef = 2.0 ** -15 if tc else gamma(C / 2 + 4)
    dl = coef * math.log2(math.e) / math.sqrt(C) * S.max(-1)
    logit = np.einsum("ojc,otc->ojt", q, K) * math.log2(math.e) / math.sqrt(C)
    spread = logit.max(-1) - logit.min(-1)
    e_p = math.log(2) * (2 * dl + U * spread) + 16 * U
    vmax = np.abs(V).max(axis=1)[:, None, :]                              # [O, 1, C]
    return (2 * e_p[..., None] + gamma(72 + splits) + (2.0 ** -15 if tc else 0.0)) * vmax


def uses_tensor_cores(kq, group):
    """The dispatcher's rule: 2- and 4-bit caches read by 8 query heads per KV
    slice take the tensor-core kernel."""
    return kq.bits in (2, 4) and group == 8


def run_case(b, shape, group, kq, vq, seed, kind="normal"):
    import torch
    outer, T, C = shape
    rng = np.random.default_rng(seed)
    if kind == "normal":
        xk = W.random_kv(rng, shape)
        xv = W.random_kv(rng, shape)
    elif kind == "peaked":                  # a few dominant keys
        xk = (rng.standard_normal(shape) * 0.2).astype(np.float32)
        xk[:, rng.integers(0, T, 3), :] *= 40.0
        xv = rng.standard_normal(shape).astype(np.float32)
    else:                                   # "offset": values near +100, zero points far below 0
        xk = (W.random_kv(rng, shape) + 100.0).astype(np.float32)
        xv = (W.random_kv(rng, shape) + 100.0).astype(np.float32)
    xk, xv = W.to_bf16_bits(xk), W.to_bf16_bits(xv)
    q = rng.standard_normal((outer, group, C)).astype(np.float32)
    qk, qv = O.quantize(xk, O.BF16, kq), O.quantize(xv, O.BF16, vq)
    K = O.dequantize_f64(qk, shape, kq, O.BF16)
    V = O.dequantize_f64(qv, shape, vq, O.BF16)
    want = O.attend(q.astype(np.float64), K, V)

    dk, dv = upload(qk), upload(qv)
    qd = torch.from_numpy(q).cuda()
    g = Guarded()                      # canary bytes around the output and the workspace
    out = g.alloc(outer * group * C * 4).view(torch.float32).view(outer, group, C)
    out.fill_(float("nan"))
    wB = b.kvq_attend_workspace(shape, group)
    ws = g.alloc(wB)
    b.kvq_attend_decode(qd, group, *dk, kq_of(b, kq), *dv, kq_of(b, vq), shape, out, ws, wB)
    g.check("kvq_attend_decode")
    got = out.cpu().numpy().astype(np.float64)
    tol = bound(q.astype(np.float64), K, V, splits=-(-T // 256), tc=uses_tensor_cores(kq, group))
    err = np.abs(got - want)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"max err {err.max():.3e}, worst err/tol {(err / tol).max():.3f}"
    return float(np.where(tol > 0, err / np.where(tol > 0, tol, 1), 0).max())


KIVI_K = O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=64, residual=128, scale_dtype=O.BF16, zero_dtype=O.BF16)
KIVI_V = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=128, scale_dtype=O.BF16, zero_dtype=O.BF16)

CASES = [
    # (outer, T), group, K format, V format
    ((4, 1000), 1, KIVI_K, KIVI_V),
    ((4, 1000), 2, KIVI_K, KIVI_V),
    ((2, 1000), 4, KIVI_K, KIVI_V),
    ((2, 1000), 8, KIVI_K, KIVI_V),
    ((3, 777), 1, O.QParams.sym(8, axis=O.ALONG_T, group=32), O.QParams.sym(8, axis=O.ALONG_C, group=128)),
    ((2, 300), 4, O.QParams.sym(2, axis=O.ALONG_T, group=0, residual=5, scale_dtype=O.BF16),
     O.QParams.sym(2, axis=O.ALONG_C, group=32, residual=5, scale_dtype=O.BF16)),
    ((2, 513), 2, O.QParams.asym(8, -128, 127, axis=O.ALONG_T, group=128, residual=17, zero_dtype=O.I8),
     O.QParams.asym(8, -128, 127, axis=O.ALONG_C, group=64, residual=17, zero_dtype=O.I8)),
    ((2, 150), 1, O.QParams.sym(4, axis=O.ALONG_T, group=64, residual=200),
     O.QParams.sym(4, axis=O.ALONG_C, group=128, residual=200)),
    ((3, 1), 8, O.QParams.sym(4, axis=O.ALONG_T, group=32), O.QParams.sym(4, axis=O.ALONG_C, group=32)),
    ((1, 4100), 4, O.QParams.asym(4, -8, 7, axis=O.ALONG_T, group=96, residual=3, zero_dtype=O.F32),
     O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=3, zero_dtype=O.F32)),
    # 8 query heads: the tensor-core kernel (2- and 4-bit), every V group size,
    # symmetric (two's complement) and signed asymmetric codes, a tile that
    # straddles the residual window, T a multiple of 16 and not
    ((2, 300), 8, O.QParams.sym(2, axis=O.ALONG_T, group=0, residual=5, scale_dtype=O.BF16),
     O.QParams.sym(2, axis=O.ALONG_C, group=32, residual=5, scale_dtype=O.BF16)),
    ((2, 700), 8, O.QParams.sym(4, axis=O.ALONG_T, group=32, residual=64),
     O.QParams.sym(4, axis=O.ALONG_C, group=128, residual=64)),
    ((1, 4100), 8, O.QParams.asym(4, -8, 7, axis=O.ALONG_T, group=96, residual=3, zero_dtype=O.F32),
     O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=3, zero_dtype=O.F32)),
    ((2, 1024), 8, O.QParams.asym(2, 0, 3, axis=O.ALONG_T, group=64, residual=0, scale_dtype=O.BF16, zero_dtype=O.BF16),
     O.QParams.asym(2, 0, 3, axis=O.ALONG_C, group=64, residual=0, scale_dtype=O.BF16, zero_dtype=O.BF16)),
]


@pytest.mark.parametrize("case", CASES, ids=str)
def test_attend_matches_oracle(b, case):
    (outer, T), group, kq, vq = case
    run_case(b, (outer, T, 128), group, kq, vq, zlib.crc32(repr(case).encode()))


def test_attend_peaked_scores(b):
    """A few keys 40x larger: nearly one-hot weights, large logit spread."""
    run_case(b, (2, 2000, 128), 2, KIVI_K, KIVI_V, 7, kind="peaked")
    run_case(b, (2, 2000, 128), 8, KIVI_K, KIVI_V, 8, kind="peaked")


def test_attend_large_offsets_take_the_exact_path(b):
    """Caches whose values sit near +100: the asymmetric zero points fall far
    below 0, outside the small integers bf16 holds exactly, and the tiles
    concerned take the float32 path of the 8-head kernel; 1 head for the
    CUDA-core kernel."""
    for group in (8, 1):
        run_case(b, (2, 600, 128), group, KIVI_K, KIVI_V, 9 + group, kind="offset")


def test_attend_kivi_workload_full_size(b):
    """The KIVI INT4 workload at full size (batch 8 x 8 KV heads, T 8192,
    128-token residual), one query per KV head, every output checked."""
    run_case(b, (64, 8192, 128), 1, KIVI_K, KIVI_V, 2)


def test_attend_empty_outer(b):
    import torch
    shape = (0, 64, 128)
    q = torch.zeros((0, 1, 128), dtype=torch.float32, device="cuda")
    out = torch.zeros((0, 1, 128), dtype=torch.float32, device="cuda")
    e = torch.zeros(16, dtype=torch.uint8, device="cuda")
    kq, vq = kq_of(b, KIVI_K), kq_of(b, KIVI_V)
    b.kvq_attend_decode(q, 1, e, e, e, e, kq, e, e, e, e, vq, shape, out, e, 16)
    torch.cuda.synchronize()


def test_attend_output_shift_within_value_error_bound(b):
    """The value bound of "KV cache 压缩：把历史装得更小" §"K 的误差会改变权重，V 的误差会改变
    内容" on the kernel: with the same quantized keys on both sides the weights
    agree, so y_gpu(K^, V^) - y(K^, V) = sum_i a_i dv_i up to the kernel's own
    float32 error, and its norm is at most max_i ||dv_i|| plus the norm of the
    derived tolerance.  The full KIVI workload, one query per KV head."""
    import torch
    shape = (64, 8192, 128)
    rng = np.random.default_rng(77)
    xk = W.to_bf16_bits(W.random_kv(rng, shape))
    xv = W.to_bf16_bits(W.random_kv(rng, shape))
    q = rng.standard_normal((shape[0], 1, shape[2])).astype(np.float32)
    qk, qv = O.quantize(xk, O.BF16, KIVI_K), O.quantize(xv, O.BF16, KIVI_V)
    K = O.dequantize_f64(qk, shape, KIVI_K, O.BF16)
    Vh = O.dequantize_f64(qv, shape, KIVI_V, O.BF16)
    V = O.bf16_bits_to_f32(xv).astype(np.float64)
    y_exact_v = O.attend(q.astype(np.float64), K, V)

    dk, dv = upload(qk), upload(qv)
    qd = torch.from_numpy(q).cuda()
    out = torch.full((shape[0], 1, shape[2]), float("nan"), dtype=torch.float32, device="cuda")
    wB = b.kvq_attend_workspace(shape, 1)
    ws = torch.empty(max(wB, 1), dtype=torch.uint8, device="cuda")
    b.kvq_attend_decode(qd, 1, *dk, kq_of(b, KIVI_K), *dv, kq_of(b, KIVI_V), shape, out, ws, wB)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    tol = bound(q.astype(np.float64), K, Vh, splits=-(-shape[1] // 256), tc=uses_tensor_cores(KIVI_K, 1))
    dy = np.linalg.norm(got - y_exact_v, axis=-1)                       # [O, 1]
    dv_max = np.linalg.norm(Vh - V, axis=-1).max(axis=1)[:, None]       # [O, 1]
    assert np.all(np.isfinite(got))
    assert np.all(dy <= dv_max + np.linalg.norm(tol, axis=-1)), f"worst ratio {(dy / dv_max).max():.3f}"
    assert dy.max() > 0
