"""How the error of a quantized cache reaches attention ("KV cache 压缩：把历史装得更小",
§"K 的误差会改变权重，V 的误差会改变内容").

The page gives two bounds and a procedure:
 - a key error dk_i moves the logit q.k_i / sqrt(d) by at most
   ||q|| ||dk_i|| / sqrt(d) (Cauchy-Schwarz);
 - with the weights held fixed (a_i >= 0, summing to 1) a value error moves
   y = sum_i a_i v_i by at most max_i ||dv_i||; when K changes too, the change
   of the weights has to be counted as well;
 - quantize K and V separately and compare logits and outputs to find the
   sensitive path.
These checks run that procedure on the oracle's quantizers and attention (CPU,
binary64).  The second bound is also checked on the GPU kernel's output in
test_attend_gpu.py.  Besides checking the bounds, the equality cases pin the
oracle's attention: weights that sum to one, logits scaled by 1/sqrt(d).
"""
import math

import numpy as np
import pytest

import oracle as O
from kv_cache_quantization_kvq_gb300 import workloads as W

SHAPE = (3, 300, 128)
FORMATS_K = [
    O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=64, residual=44, scale_dtype=O.BF16, zero_dtype=O.BF16),
    O.QParams.sym(8, axis=O.ALONG_T, group=0),
    O.QParams.sym(2, axis=O.ALONG_T, group=32, residual=7, scale_dtype=O.BF16),
]
FORMATS_V = [
    O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=44, scale_dtype=O.BF16, zero_dtype=O.BF16),
    O.QParams.sym(8, axis=O.ALONG_C, group=128),
    O.QParams.sym(2, axis=O.ALONG_C, group=32, residual=7, scale_dtype=O.BF16),
]


def cache(seed):
    rng = np.random.default_rng(seed)
    xk = W.to_bf16_bits(W.random_kv(rng, SHAPE))
    xv = W.to_bf16_bits(W.random_kv(rng, SHAPE))
    q = rng.standard_normal((SHAPE[0], 4, SHAPE[2])).astype(np.float64)
    exact = lambda x: O.bf16_bits_to_f32(x).astype(np.float64)
    return q, xk, xv, exact(xk), exact(xv)


def dequant(x_bits, qp):
    return O.dequantize_f64(O.quantize(x_bits, O.BF16, qp), SHAPE, qp, O.BF16)


def logits(q, K):
    return np.einsum("ojc,otc->ojt", q, K) / math.sqrt(K.shape[-1])


@pytest.mark.parametrize("fi", range(len(FORMATS_K)))
def test_logit_shift_within_key_error_bound(fi):
    """|q.dk_i| / sqrt(d) <= ||q|| ||dk_i|| / sqrt(d) for every query and token;
    residual tokens (exact) do not move.  Catches a logit scaled by anything
    but 1/sqrt(d) on one side only."""
    qp = FORMATS_K[fi]
    q, xk, _, K, _ = cache(10 + fi)
    Kh = dequant(xk, qp)
    dl = logits(q, Kh) - logits(q, K)
    dk = np.linalg.norm(Kh - K, axis=-1)                               # [O, T]
    bound = np.linalg.norm(q, axis=-1)[..., None] * dk[:, None, :] / math.sqrt(SHAPE[2])
    assert np.all(np.abs(dl) <= bound * (1 + 1e-12) + 1e-300)
    R = qp.residual
    if R:
        assert np.all(dl[:, :, SHAPE[1] - R:] == 0.0)
    # equality case: a query parallel to one token's key error
    j = int(np.argmax(dk[0, : SHAPE[1] - R]))
    qj = (Kh - K)[0, j][None, None, :] * 3.0
    lhs = abs(float(logits(qj, Kh[:1])[0, 0, j] - logits(qj, K[:1])[0, 0, j]))
    rhs = float(np.linalg.norm(qj) * dk[0, j] / math.sqrt(SHAPE[2]))
    assert rhs > 0 and abs(lhs - rhs) <= 1e-12 * rhs


@pytest.mark.parametrize("fi", range(len(FORMATS_V)))
def test_output_shift_within_value_error_bound(fi):
    """Weights fixed (same K on both sides): ||y(K, V^) - y(K, V)|| <= max_i
    ||dv_i||.  Catches weights that do not sum to one or go negative."""
    qp = FORMATS_V[fi]
    q, _, xv, K, V = cache(20 + fi)
    Vh = dequant(xv, qp)
    dy = np.linalg.norm(O.attend(q, K, Vh) - O.attend(q, K, V), axis=-1)   # [O, G]
    dv_max = np.linalg.norm(Vh - V, axis=-1).max(axis=1)                    # [O]
    assert np.all(dy <= dv_max[:, None] * (1 + 1e-12))
    assert dy.max() > 0


def test_output_shift_equals_a_common_value_error():
    """The bound's equality case: the same error c on every value row moves
    the output by exactly c, whatever the weights -- only weights that sum to
    one do that."""
    q, _, _, K, V = cache(30)
    c = np.random.default_rng(31).standard_normal(SHAPE[2])
    dy = O.attend(q, K, V + c) - O.attend(q, K, V)
    assert np.allclose(dy, np.broadcast_to(c, dy.shape), rtol=0, atol=1e-12 * np.abs(c).max() * 64)


@pytest.mark.parametrize("fi", range(len(FORMATS_K)))
def test_k_and_v_quantized_separately(fi):
    """The page's procedure: quantize K only, V only, then both.
     - V only: the output moves within the value bound above.
     - K only: with every logit moved by at most delta (the key bound), each
       weight moves by a factor in [e^-2delta, e^2delta], so
       ||dy|| <= (e^(2 delta) - 1) max_i ||v_i||.
     - both: within the sum of the two.
    Catches a softmax that is not shift-invariant or weights computed from
    anything but the logits."""
    kq, vq = FORMATS_K[fi], FORMATS_V[fi]
    q, xk, xv, K, V = cache(40 + fi)
    Kh, Vh = dequant(xk, kq), dequant(xv, vq)
    y = O.attend(q, K, V)
    dk = np.linalg.norm(Kh - K, axis=-1).max(axis=1)                        # [O]
    delta = np.linalg.norm(q, axis=-1) * dk[:, None] / math.sqrt(SHAPE[2])  # [O, G]
    vmax = np.linalg.norm(V, axis=-1).max(axis=1)[:, None]
    k_bound = np.expm1(2 * delta) * vmax
    v_bound = np.linalg.norm(Vh - V, axis=-1).max(axis=1)[:, None]
    dy_k = np.linalg.norm(O.attend(q, Kh, V) - y, axis=-1)
    dy_v = np.linalg.norm(O.attend(q, K, Vh) - y, axis=-1)
    dy_kv = np.linalg.norm(O.attend(q, Kh, Vh) - y, axis=-1)
    slack = 1 + 1e-9
    assert np.all(dy_k <= k_bound * slack)
    assert np.all(dy_v <= v_bound * slack)
    # y(K^, V^) - y = [y(K^, V^) - y(K^, V)] + [y(K^, V) - y]: value bound + key bound
    assert np.all(dy_kv <= (v_bound + k_bound) * slack)
    assert dy_k.max() > 0 and dy_v.max() > 0
