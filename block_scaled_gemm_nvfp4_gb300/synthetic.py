"""Seeded synthetic inputs shaped like the pages' layers.

This module only draws random BF16 tensors; it holds none of the NVFP4
arithmetic and is shared by the tests, the smoke check and the benchmark so
that the GPU path and the oracle see identical inputs.

The pages train on private corpora (a 10T-token blend for the 12B hybrid
Mamba-Transformer in "NVFP4 Treina com Precisao de 16 Bits...", and a
64B-token corpus for the 3B model in "Full-Stack FP4...", section 4); neither
is needed for the linear layer's arithmetic, so normal draws with the layer
shapes stand in for them.

Seeds: ``seed_for(config, tensor) = 20260811 + 100 * config + tensor``.
"""
import numpy as np
import torch

BASE_SEED = 20260811


def seed_for(config: int, tensor: int) -> int:
    return BASE_SEED + 100 * config + tensor


def normal_bf16(shape, std=1.0, seed=0) -> torch.Tensor:
    """i.i.d. N(0, std^2), drawn in FP32 and rounded to BF16 (RNE)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


def normal_with_outliers_bf16(shape, frac=1e-3, factor=100.0, seed=0) -> torch.Tensor:
    """N(0,1) with a seeded uniform sample (without replacement) of
    ``frac`` of the positions multiplied by ``factor``."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32)
    n = a.size
    k = int(round(n * frac))
    if k:
        idx = rng.choice(n, size=k, replace=False)
        a.reshape(-1)[idx] *= np.float32(factor)
    return torch.from_numpy(a).to(torch.bfloat16)


def channel_scaled_bf16(shape, lo=1e-2, hi=10.0, seed=0) -> torch.Tensor:
    """N(0,1) times a per-column factor drawn log-uniform in [lo, hi]."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32)
    c = np.exp(rng.uniform(np.log(lo), np.log(hi), size=(shape[-1],))).astype(np.float32)
    a *= c[None, :]
    return torch.from_numpy(a).to(torch.bfloat16)


def as_u16(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor (CPU) -> numpy uint16 bit patterns, same shape."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# --- the workloads -----------------------------------------------------------
# Config 0: one small linear fprop (256x256 operands).
def config0():
    x = normal_bf16((256, 256), seed=seed_for(0, 0))
    w = normal_bf16((256, 256), seed=seed_for(0, 1))
    return x, w


# Config 1: quantise-only sweep tensors.
QUANT_SWEEP_SHAPES = [(4096, 5120), (8192, 20480)]


def config1(shape_idx: int):
    return normal_with_outliers_bf16(QUANT_SWEEP_SHAPES[shape_idx], seed=seed_for(1, shape_idx))


# Config 2: 12B-hybrid-shaped MLP up-projection (tokens 8192 = 4 x 2048,
# hidden 5120, FFN 20480).
MLP12B = dict(tokens=8192, hidden=5120, ffn=20480)


def config2(tokens=8192, hidden=5120, ffn=20480):
    x = normal_bf16((tokens, hidden), seed=seed_for(2, 0))
    w = normal_bf16((ffn, hidden), std=0.02, seed=seed_for(2, 1))
    dy = normal_bf16((tokens, ffn), std=1e-3, seed=seed_for(2, 2))
    return x, w, dy


# Config 3: 3B-shaped projections, tokens 16384, hidden 3072.
PROJ3B = [("qkv", 3072, 9216), ("mlp_up", 3072, 8192), ("mlp_down", 8192, 3072)]


def config3(name: str, tokens=16384):
    idx = [p[0] for p in PROJ3B].index(name)
    _, din, dout = PROJ3B[idx]
    x = channel_scaled_bf16((tokens, din), seed=seed_for(3, 3 * idx + 0))
    w = normal_bf16((dout, din), std=0.02, seed=seed_for(3, 3 * idx + 1))
    dy = channel_scaled_bf16((tokens, dout), seed=seed_for(3, 3 * idx + 2))
    return x, w, dy


# Config 4: GEMM roofline probes.
def config4(m, n, k):
    a = normal_bf16((m, k), seed=seed_for(4, 0))
    b = normal_bf16((n, k), seed=seed_for(4, 1))
    return a, b
