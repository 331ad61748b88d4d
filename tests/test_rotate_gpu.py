"""CUDA randomized Hadamard rotation vs the CPU oracle (binary64 matrix
product with the Sylvester matrix).

Tolerance, derived from the kernel's float32 arithmetic (u = 2^-24,
gamma_n = n u / (1 - n u)): every output is built by log2(C) butterfly
additions whose partial sums are bounded by sum_c |x_c|, then one multiply by
the rounded 1/sqrt(C):  |y - y_ref| <= B = gamma_{log2 C + 2} sum_c |x_c| / sqrt(C).
A bf16 output adds its own rounding: |y - y_ref| <= 2^-8 (|y_ref| + B) + B.
"""
import math
import zlib

import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, kb
from kv_cache_quantization_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def b():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kb()


def tol(x64, ref, out_bf16):
    C = x64.shape[-1]
    n = int(math.log2(C)) + 2
    B = (n * U / (1 - n * U)) * np.abs(x64).sum(-1, keepdims=True) / math.sqrt(C)
    return 2.0 ** -8 * (np.abs(ref) + B) + B if out_bf16 else B


def run(b, shape, C, x_bf16, out_bf16, inverse, seed, inplace=False):
    import torch
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(shape + (C,)) * np.exp(rng.uniform(-3, 3, shape + (1,)))).astype(np.float32)
    if x_bf16:
        bits = W.to_bf16_bits(x)
        x64 = O.bf16_bits_to_f32(bits).astype(np.float64)
        xd = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        x64 = x.astype(np.float64)
        xd = torch.from_numpy(x).cuda()
    s = np.where(rng.random(C) < 0.5, -1, 1).astype(np.int8)
    sd = torch.from_numpy(s).cuda()
    ref = O.rotate(x64, s, inverse=inverse)
    od = b.BF16 if out_bf16 else b.F32
    g = Guarded()                      # canary bytes around the output
    if inplace:
        out = xd
    else:
        tdt = torch.bfloat16 if out_bf16 else torch.float32
        out = g.alloc(x.size * (2 if out_bf16 else 4)).view(tdt).view(xd.shape)
    got = b.rotate(xd, sd, inverse=inverse, out=out, out_dtype=od)
    g.check("kvq_rotate")
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    assert np.all(err <= tol(x64, ref, out_bf16)), f"max err {err.max():.3e}"


@pytest.mark.parametrize("C", [32, 64, 128, 256, 512, 1024])
@pytest.mark.parametrize("dtypes", [(True, True), (True, False), (False, False), (False, True)], ids=str)
@pytest.mark.parametrize("inverse", [False, True])
def test_rotate_matches_oracle(b, C, dtypes, inverse):
    run(b, (3, 37), C, dtypes[0], dtypes[1], inverse, zlib.crc32(repr((C, dtypes, inverse)).encode()))


@pytest.mark.parametrize("C", [64, 128])
def test_rotate_in_place(b, C):
    run(b, (2, 21), C, True, True, False, C, inplace=True)
    run(b, (2, 21), C, False, False, True, C + 1, inplace=True)


def test_rotate_round_trip_on_device(b):
    """forward then inverse on the GPU in float32 returns x within twice the bound."""
    import torch
    rng = np.random.default_rng(60)
    x = rng.standard_normal((4, 100, 128)).astype(np.float32)
    s = torch.from_numpy(np.where(rng.random(128) < 0.5, -1, 1).astype(np.int8)).cuda()
    xd = torch.from_numpy(x).cuda()
    back = b.rotate(b.rotate(xd, s), s, inverse=True)
    torch.cuda.synchronize()
    x64 = x.astype(np.float64)
    assert np.all(np.abs(back.cpu().numpy() - x64) <= 3 * tol(x64, x64, False))


def test_rotate_kivi_keys_sampled_rows(b):
    """The KIVI key cache at full size (bf16 [64, 8192, 128]), bf16 -> bf16:
    2000 sampled rows against the oracle."""
    import torch
    K, _ = W.kivi_kv("cuda", seed=2)
    rng = np.random.default_rng(61)
    s_np = np.where(rng.random(128) < 0.5, -1, 1).astype(np.int8)
    out = b.rotate(K, torch.from_numpy(s_np).cuda())
    torch.cuda.synchronize()
    flat_in = K.reshape(-1, 128)
    idx = torch.from_numpy(rng.choice(flat_in.shape[0], 2000, replace=False)).cuda()
    xs = flat_in[idx].float().cpu().numpy().astype(np.float64)
    ref = O.rotate(xs, s_np)
    got = out.reshape(-1, 128)[idx].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol(xs, ref, True))
