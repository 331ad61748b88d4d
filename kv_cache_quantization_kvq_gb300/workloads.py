"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers; it holds none of the compression
method's arithmetic.  Both the tests / benchmark (for the CUDA path) and the
CPU oracle consume the SAME buffers produced here: small cases are drawn with
numpy on the host, large ones with a seeded torch generator on the device and
copied to the host when the oracle needs them.

Workloads (no dataset is involved; these stand in for the KV caches and
attention histories of LLMs that the pages discuss):
  tiny      K-like fp32 [1, 256, 128], N(0,1) with 4 outlier channels x10;
            attention history [1, 32, 256], rows softmax(2 * N(0,1)).
  kivi      bf16 K, V [batch*heads, T, 128], N(0,1); 2 % of the K channels
            (per batch, head, dim) scaled x8 over all tokens.
  fullmodel bf16 K, V [layers, T, heads*128]: per channel a Student-t
            (nu = 4) normalised to unit variance, times a per-channel std
            drawn log-uniformly from [0.1, 10].
  sweep     bf16 K, V [batch*heads, T, 128], N(0,1) with i.i.d. 1 % of the
            elements scaled x20.
  eviction  fp32 history [heads, steps, T]: each row softmax(3 * Gumbel(0,1)
            + 4 on 256 planted tokens per head, drawn without replacement from
            [0, T - window) and shared by all steps); bf16 K, V [heads, T, 128]
            N(0,1).
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------- small, host

def tiny_inputs(seed: int = 0):
    """(x [1, 256, 128] float32, hist [1, 32, 256] float32)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((256, 128), dtype=np.float32)
    ch = rng.choice(128, 4, replace=False)
    x[:, ch] *= 10.0
    z = rng.standard_normal((32, 256)) * 2.0
    e = np.exp(z - z.max(axis=1, keepdims=True))
    hist = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return x.reshape(1, 256, 128), hist.reshape(1, 32, 256)


def random_kv(rng: np.random.Generator, shape, outlier_frac=0.02, outlier_scale=8.0):
    """float32 [outer, T, C] N(0,1) with a fraction of (outer, channel) columns scaled."""
    x = rng.standard_normal(shape, dtype=np.float32)
    outer, T, C = shape
    n = int(round(outlier_frac * outer * C))
    if n and T:
        idx = rng.choice(outer * C, n, replace=False)
        x[idx // C, :, idx % C] *= outlier_scale
    return x


def random_history(rng: np.random.Generator, heads, steps, T, temp=3.0, planted=8, boost=4.0, window=0):
    """float32 [heads, steps, T]: row softmax of temp*Gumbel + boost on planted tokens."""
    u = rng.random((heads, steps, T))
    g = -np.log(-np.log(np.clip(u, 1e-300, None)))
    logits = temp * g
    hi = max(T - window, 0)
    for h in range(heads):
        if hi > 0:
            p = rng.choice(hi, min(planted, hi), replace=False)
            logits[h, :, p] += boost
    logits -= logits.max(axis=-1, keepdims=True)
    e = np.exp(logits)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), rounded by torch (input preparation only)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- large, device

def _gen(device, seed):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def kivi_kv(device="cuda", seed=2, batch=8, heads=8, T=8192, D=128, outlier_frac=0.02, outlier_scale=8.0):
    """bf16 (K, V) [batch*heads, T, D]."""
    import torch
    g = _gen(device, seed)
    outer = batch * heads
    K = torch.randn((outer, T, D), generator=g, device=device, dtype=torch.float32)
    V = torch.randn((outer, T, D), generator=g, device=device, dtype=torch.float32)
    n = int(round(outlier_frac * outer * D))
    if n:
        idx = torch.randperm(outer * D, generator=g, device=device)[:n]
        K.view(outer, T, D)[idx // D, :, idx % D] *= outlier_scale
    return K.to(torch.bfloat16), V.to(torch.bfloat16)


def fullmodel_kv(device="cuda", seed=3, layers=32, T=8192, heads=32, D=128):
    """bf16 (K, V) [layers, T, heads*D], per-channel scaled Student-t(4)."""
    import torch
    g = _gen(device, seed)
    C = heads * D
    out = []
    for _ in range(2):
        t = torch.empty((layers, T, C), device=device, dtype=torch.bfloat16)
        for l in range(layers):
            sig = torch.exp(torch.empty(C, device=device).uniform_(math.log(0.1), math.log(10.0), generator=g))
            z = torch.randn((T, C), generator=g, device=device)
            u1 = torch.rand((T, C), generator=g, device=device).clamp_min_(1e-30)
            u2 = torch.rand((T, C), generator=g, device=device).clamp_min_(1e-30)
            chi2_4 = -2.0 * (torch.log(u1) + torch.log(u2))          # chi-square, 4 dof
            student = z / torch.sqrt(chi2_4 / 4.0)                    # t, 4 dof (variance 2)
            t[l] = (student / math.sqrt(2.0) * sig).to(torch.bfloat16)
        out.append(t)
    return out[0], out[1]


def sweep_kv(device="cuda", seed=4, batch=16, heads=8, T=32768, D=128, p=0.01, scale=20.0):
    """bf16 (K, V) [batch*heads, T, D], N(0,1) with Bernoulli(p) elements x scale."""
    import torch
    g = _gen(device, seed)
    out = []
    for _ in range(2):
        x = torch.randn((batch * heads, T, D), generator=g, device=device)
        m = torch.rand((batch * heads, T, D), generator=g, device=device) < p
        x = torch.where(m, x * scale, x)
        out.append(x.to(torch.bfloat16))
        del x, m
    return out[0], out[1]


def eviction_inputs(device="cuda", seed=5, heads=32, steps=64, T=131072, D=128, planted=256, window=128,
                    boost=4.0, temp=3.0, with_kv=True):
    """(hist fp32 [heads, steps, T], K bf16 [heads, T, D], V bf16 [heads, T, D])."""
    import torch
    g = _gen(device, seed)
    hist = torch.empty((heads, steps, T), device=device, dtype=torch.float32)
    for h in range(heads):
        u = torch.rand((steps, T), generator=g, device=device).clamp_(1e-30, 1.0 - 1e-7)
        logits = temp * (-torch.log(-torch.log(u)))
        hi = max(T - window, 0)
        if hi:
            p = torch.randperm(hi, generator=g, device=device)[:min(planted, hi)]
            logits[:, p] += boost
        hist[h] = torch.softmax(logits, dim=-1)
    if not with_kv:
        return hist, None, None
    K = torch.randn((heads, T, D), generator=g, device=device).to(torch.bfloat16)
    V = torch.randn((heads, T, D), generator=g, device=device).to(torch.bfloat16)
    return hist, K, V
