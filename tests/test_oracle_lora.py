"""Pins for the oracle's LoRA-SVD projection forward (CPU only).

Checked against facts fixed outside the oracle's code:
  * with beta = 0 it is the NVFP4 GEMM of X and W_res;
  * with every W_res code zero and small-integer BF16 inputs (every product
    and sum exact) it is beta * X L1^T L2^T in integer arithmetic;
  * where X L1^T is not a BF16 value, the branch rounds it to BF16 first
    (torch's float64 matmul and bfloat16 conversion as the restatement).
"""
import numpy as np
import torch

import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn


def _bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _quant(x_u16, **cfg):
    return oracle.quantize(x_u16, oracle.make_cfg(**cfg))


def test_beta_zero_is_the_nvfp4_gemm():
    x = syn.as_u16(syn.normal_bf16((32, 64), seed=1))
    w = syn.as_u16(syn.normal_bf16((48, 64), seed=2, std=0.02))
    l1 = syn.as_u16(syn.normal_bf16((16, 64), seed=3))
    l2 = syn.as_u16(syn.normal_bf16((48, 16), seed=4))
    xq, wq = _quant(x), _quant(w, block=1)
    y = oracle.lora_forward(xq, wq, x, l1, l2, 0.0)
    assert np.array_equal(y, oracle.gemm_f64(xq, wq, 32, 48, 64))


def test_low_rank_branch_exact_on_integers():
    rng = np.random.default_rng(5)
    T, din, dout, r = 16, 32, 32, 8
    xi = rng.integers(-3, 4, size=(T, din))
    l1i = rng.integers(-2, 3, size=(r, din))
    l2i = rng.integers(-2, 3, size=(dout, r))
    x, l1, l2 = (_bits(torch.from_numpy(a.astype(np.float32))) for a in (xi, l1i, l2i))
    zero_w = (np.zeros((dout, din // 2), np.uint8), np.full((dout, din // 16), 0x38, np.uint8), np.float32(1.0))
    xq = _quant(x)
    y = oracle.lora_forward(xq, zero_w, x, l1, l2, 0.5)
    ref = 0.5 * (xi @ l1i.T) @ l2i.T  # |X L1^T| <= 96: exact in BF16
    assert np.array_equal(y, ref.astype(np.float64))


def test_branch_rounds_its_intermediate_to_bf16():
    x = syn.as_u16(syn.normal_bf16((8, 32), seed=6))
    l1 = syn.as_u16(syn.normal_bf16((4, 32), seed=7))
    l2 = syn.as_u16(syn.normal_bf16((16, 4), seed=8))
    zero_w = (np.zeros((16, 16), np.uint8), np.zeros((16, 2), np.uint8), np.float32(1.0))
    y = oracle.lora_forward(_quant(x), zero_w, x, l1, l2, 2.0)
    f = lambda u: torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).double()  # noqa: E731
    u = (f(x) @ f(l1).T).to(torch.bfloat16).double()
    ref = 2.0 * (u @ f(l2).T)
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=0)
    # and the rounding matters: without it the result differs
    unrounded = 2.0 * ((f(x) @ f(l1).T) @ f(l2).T)
    assert not np.allclose(y, unrounded.numpy(), rtol=1e-9, atol=0)


def test_down_step_is_the_bf16_rounded_fp64_product():
    x = syn.as_u16(syn.normal_bf16((24, 96), seed=9))
    l1 = syn.as_u16(syn.normal_bf16((40, 96), seed=10))
    u, ue = oracle.lora_down(x, l1)
    f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double()  # noqa: E731
    ref = f(x) @ f(l1).T
    assert np.allclose(ue, ref.numpy(), rtol=1e-13, atol=0)
    assert np.array_equal(u, _bits(ref.float()))


def test_sampled_forward_equals_full_forward():
    x = syn.as_u16(syn.normal_bf16((48, 64), seed=11))
    w = syn.as_u16(syn.normal_bf16((80, 64), seed=12, std=0.02))
    l1 = syn.as_u16(syn.normal_bf16((16, 64), seed=13))
    l2 = syn.as_u16(syn.normal_bf16((80, 16), seed=14))
    xq, wq = _quant(x), _quant(w, block=1)
    full = oracle.lora_forward(xq, wq, x, l1, l2, 0.75)
    rng = np.random.default_rng(15)
    t = rng.integers(0, 48, size=200)
    n = rng.integers(0, 80, size=200)
    assert np.array_equal(oracle.lora_forward_sampled(xq, wq, x, l1, l2, 0.75, t, n), full[t, n])
