"""Pins for the oracle's delayed-scaling quantiser (CPU only).

The tensor scale comes from a supplied amax instead of the operand's own.
Checked against facts fixed outside the oracle's code:
  * with the operand's own amax (found here with numpy) it is the ordinary
    quantisation;
  * multiplying the supplied amax by 4 (exact in FP32) divides every normal
    block scale by 4 (two E4M3 exponent steps) and leaves the codes alone;
  * a brute-force restatement with numpy FP32 arithmetic, torch's E4M3
    conversion and a nearest-grid search with ties to the even code gives
    the same bytes, including blocks whose scale saturates at 448 and
    elements that saturate at 6 when the supplied amax is too small.
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _f32(x_u16):
    return (x_u16.astype(np.uint32) << 16).view(np.float32)


def _e4m3_rne_sat(t):
    # RNE to E4M3 with saturation: anything at or above 448 is 448 (the next
    # E4M3 step would be 480, so clamping first gives the same byte).
    t = np.minimum(t.astype(np.float32), np.float32(448.0))
    return torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_value(b):
    return torch.from_numpy(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _e2m1_rne_brute(v):
    # nearest of the eight magnitudes, ties to the even code, |v| > 6 -> 6;
    # the sign bit of v is kept (negative zero gives code 8)
    mag = np.abs(v.astype(np.float64))
    d = np.abs(mag[..., None] - GRID)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # among tied candidates take the even code (codes 0..7 index GRID)
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    return (code | (np.signbit(v) * 8)).astype(np.uint8)


def _brute_quantize(x_u16, amax):
    x = _f32(x_u16)
    rows, cols = x.shape
    s = np.float32(amax) / np.float32(2688.0)
    if s == 0:
        s = np.float32(1.0)
    blocks = x.reshape(rows, cols // 16, 16)
    bamax = np.abs(blocks).max(axis=2).astype(np.float32)
    t = (bamax / np.float32(6.0)) / s
    sf = _e4m3_rne_sat(t)
    denom = _e4m3_value(sf) * s
    with np.errstate(divide="ignore", invalid="ignore"):
        v = blocks / denom[..., None]
    codes = _e2m1_rne_brute(v)
    codes[sf == 0] = 0
    codes = codes.reshape(rows, cols)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf, s


def test_own_amax_is_ordinary_quantisation():
    x = syn.as_u16(syn.normal_with_outliers_bf16((96, 256), frac=0.01, seed=31))
    amax = np.abs(_f32(x)).max()
    for cfg in (oracle.make_cfg(), oracle.make_cfg(block=1), oracle.make_cfg(transpose=1, rounding=1, sr_seed=3)):
        a = oracle.quantize(x, cfg)
        b = oracle.quantize_given_amax(x, cfg, amax)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]
    assert b[2] == np.float32(amax) / np.float32(2688.0)


def test_four_times_the_amax_shifts_normal_scales_two_steps():
    x = syn.as_u16(syn.normal_bf16((64, 512), seed=32))
    amax = np.abs(_f32(x)).max()
    c1, s1, t1 = oracle.quantize_given_amax(x, oracle.make_cfg(), amax)
    c4, s4, t4 = oracle.quantize_given_amax(x, oracle.make_cfg(), amax * 4)
    assert t4 == t1 * 4
    ok = _e4m3_value(s1) >= 2.0 ** -4  # stays normal after two exponent steps down
    assert ok.mean() > 0.9
    assert np.array_equal(s4[ok], s1[ok] - 0x10)
    rows_ok = np.repeat(ok, 8, axis=1)  # 8 code bytes per block
    assert np.array_equal(c4[rows_ok], c1[rows_ok])


@pytest.mark.parametrize("factor", [1.0, 3.0, 0.25, 1.0 / 64])
def test_matches_brute_force(factor):
    x = syn.as_u16(syn.normal_with_outliers_bf16((64, 320), frac=0.02, seed=33))
    amax = np.float32(np.abs(_f32(x)).max() * factor)
    codes, sf, s = oracle.quantize_given_amax(x, oracle.make_cfg(), amax)
    bc, bsf, bs = _brute_quantize(x, amax)
    assert s == bs
    assert np.array_equal(sf, bsf)
    assert np.array_equal(codes, bc)
    if factor < 1:
        # the amax is too small: some scales stop at 448, some codes at 6
        assert (sf == 0x7E).any()
        assert ((codes & 7) == 7).any() or ((codes >> 4) & 7 == 7).any()


def test_zero_amax_gives_unit_scale():
    x = syn.as_u16(syn.normal_bf16((16, 64), seed=34))
    codes, sf, s = oracle.quantize_given_amax(x, oracle.make_cfg(), 0.0)
    assert s == 1.0
    bc, bsf, _ = _brute_quantize(x, 0.0)
    assert np.array_equal(sf, bsf) and np.array_equal(codes, bc)


def test_bad_amax_or_nonfinite_input_is_an_error():
    x = syn.as_u16(syn.normal_bf16((16, 32), seed=35)).copy()
    for bad in (float("inf"), float("nan"), -1.0):
        with pytest.raises(oracle.OracleError) as e:
            oracle.quantize_given_amax(x, oracle.make_cfg(), bad)
        assert e.value.status == oracle.ERR_NONFINITE
    x[2, 3] = 0x7F80
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize_given_amax(x, oracle.make_cfg(), 1.0)
    assert e.value.status == oracle.ERR_NONFINITE
