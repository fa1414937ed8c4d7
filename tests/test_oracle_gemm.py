"""Pins for the oracle's dequantiser and FP64 GEMM (CPU only).

Tiny GEMMs are compared with a brute-force FP64 product of the dequantised
operands computed here with numpy, and hand-built operands (every block scale
1.0, tensor scale 1) give integer multiples of 1/4, where every sum is exact.
"""
import numpy as np
import pytest

import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _pack(codes4):
    return (codes4[:, 0::2] | (codes4[:, 1::2] << 4)).astype(np.uint8)


def _grid_values(codes4):
    mag = GRID[codes4 & 7]
    return np.where(codes4 & 8, -mag, mag)


def test_dequantize_closed_form():
    rng = np.random.default_rng(0)
    c4 = rng.integers(0, 16, size=(8, 64), dtype=np.uint8)
    sf = rng.integers(0, 127, size=(8, 4), dtype=np.uint8)
    s = np.float32(0.0371)
    d = oracle.dequantize(_pack(c4), sf, s, 8, 64)
    e4 = np.vectorize(oracle.e4m3_value)(sf)
    assert np.array_equal(d, _grid_values(c4) * np.repeat(e4, 16, axis=1) * np.float64(s))


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 64), (16, 16, 96), (64, 48, 64)])
def test_tiny_gemm_matches_numpy_fp64(M, N, K):
    a = syn.as_u16(syn.normal_bf16((M, K), seed=M * 7 + K))
    b = syn.as_u16(syn.normal_bf16((N, K), seed=N * 11 + K))
    qa = oracle.quantize(a, oracle.make_cfg())
    qb = oracle.quantize(b, oracle.make_cfg(block=0, rounding=1, sr_seed=5))
    got = oracle.gemm_f64(qa, qb, M, N, K)
    da = oracle.dequantize(*qa, M, K)
    db = oracle.dequantize(*qb, N, K)
    ref = da @ db.T
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    mi = np.array([0, M - 1, M // 2])
    ni = np.array([N - 1, 0, N // 2])
    assert np.allclose(oracle.gemm_f64_sampled(qa, qb, K, mi, ni), ref[mi, ni], rtol=1e-12, atol=1e-300)


def test_unit_scales_give_exact_integer_quarters():
    rng = np.random.default_rng(1)
    M, N, K = 8, 8, 256
    ca = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
    cb = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    one = np.full((M, K // 16), 0x38, dtype=np.uint8)
    qa = (_pack(ca), one, np.float32(1.0))
    qb = (_pack(cb), one[:N], np.float32(1.0))
    got = oracle.gemm_f64(qa, qb, M, N, K)
    ref = _grid_values(ca) @ _grid_values(cb).T
    assert np.array_equal(got, ref)
    assert np.array_equal(got * 4, np.round(got * 4))
