"""Pins for the oracle's quantised AdamW state codec (CPU only).

Checked against facts fixed outside the oracle's code:
  * BF16 rounding equals torch's float32 -> bfloat16 conversion;
  * the inverse transform undoes the forward one (H16 H16 = 16 I), exactly on
    inputs whose sums are exact;
  * first moment: every block's scale byte is one of the two candidates
    E4M3((bamax/6)/s) and E4M3((bamax/4)/s), computed here with numpy FP32 and
    torch's E4M3 conversion, and it is the one whose round-to-nearest squared
    error (a brute-force nearest-grid search here) is smaller, the 6-mapping on
    a tie; stochastic rounding never leaves the bracketing grid points and the
    decoded state is unbiased over seeds;
  * second moment: the tile mean is BF16 of the exact mean where the FP32 sums
    are exact; tiles whose square roots are one BF16 value decode exactly;
    the decoded state is a square, and close to the input.
"""
import numpy as np
import pytest
import torch

import oracle

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
RS = 0x5EED
SS = 0xBEEF


def _e4m3_rne_sat(t):
    t = np.minimum(np.asarray(t, dtype=np.float32), np.float32(448.0))
    return torch.from_numpy(np.ascontiguousarray(t)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_value(b):
    return torch.from_numpy(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _rne_brute(v):
    mag = np.abs(v.astype(np.float64))
    d = np.abs(mag[..., None] - GRID)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(8) % 2 == 0)
    idx = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    return np.where(np.signbit(v), -GRID[idx], GRID[idx])


def _unpack(codes, cols):
    c = np.empty((codes.shape[0], cols), dtype=np.uint8)
    c[:, 0::2] = codes & 15
    c[:, 1::2] = codes >> 4
    mag = GRID[c & 7]
    return np.where(c & 8, -mag, mag)


def _transform(m):
    sigma = oracle.rht_signs(RS)
    x = m.astype(np.float32).reshape(-1, 16)
    return np.stack([oracle.rht16(r, sigma) for r in x]).reshape(m.shape)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-20, 20, 20000),
                        # exact ties between two BF16 values, even and odd lower neighbours
                        ((np.arange(1, 2001, dtype=np.uint32) << 16) | 0x8000).view(np.float32)])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(x) for x in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_inverse_transform():
    sigma = oracle.rht_signs(RS)
    rng = np.random.default_rng(6)
    ints = rng.integers(-64, 64, size=16).astype(np.float32)  # all sums exact
    assert np.array_equal(oracle.rht16_inverse(oracle.rht16(ints, sigma), sigma), ints)
    x = rng.standard_normal(16).astype(np.float32)
    assert np.allclose(oracle.rht16_inverse(oracle.rht16(x, sigma), sigma), x, rtol=0, atol=1e-6)


@pytest.mark.parametrize("scale", [1e-3, 1.0])
def test_m_scale_choice_is_the_better_of_4_and_6(scale):
    rng = np.random.default_rng(7)
    m = (rng.standard_normal((48, 128)) * scale).astype(np.float32)
    m[::7, ::13] *= 30  # heavy tail
    codes, sf, s = oracle.qadamw_m_encode(m, RS, SS)
    x = _transform(m)
    assert s == np.float32(np.abs(x).max()) / np.float32(2688.0)
    runs = x.reshape(-1, 16)
    bamax = np.abs(runs).max(axis=1).astype(np.float32)
    s32 = np.float32(s)
    sf6 = _e4m3_rne_sat((bamax / np.float32(6.0)) / s32)
    sf4 = _e4m3_rne_sat((bamax / np.float32(4.0)) / s32)

    def err(sfb):
        d = (_e4m3_value(sfb) * s32).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = _rne_brute((runs / d[:, None]).astype(np.float32))
        deq = np.where(sfb[:, None] == 0, 0.0, q * d[:, None]).astype(np.float32)
        e = (runs - deq).astype(np.float32)
        acc = np.zeros(len(runs), dtype=np.float32)
        for j in range(16):  # left-to-right FP32 sum
            acc = (acc + (e[:, j] * e[:, j]).astype(np.float32)).astype(np.float32)
        return acc

    pick4 = err(sf4) < err(sf6)
    assert np.array_equal(sf.reshape(-1), np.where(pick4, sf4, sf6))
    assert pick4.any() and (~pick4).any()
    # stochastic rounding stays on the bracketing grid points
    d = (_e4m3_value(sf.reshape(-1)) * s32).astype(np.float32)
    v = np.abs((runs / d[:, None]).astype(np.float64))
    q = np.abs(_unpack(codes, 128).reshape(-1, 16))
    lo = GRID[np.searchsorted(GRID, np.minimum(v, 6.0), side="right") - 1]
    hi = GRID[np.minimum(np.searchsorted(GRID, np.minimum(v, 6.0), side="right"), 7)]
    ok = (q == lo) | (q == hi) | ((v >= 6.0) & (q == 6.0))
    assert ok[sf.reshape(-1) != 0].all()


def test_m_decode_is_unbiased_over_seeds():
    rng = np.random.default_rng(8)
    m = (rng.standard_normal((16, 64)) * 1e-2).astype(np.float32)
    acc = np.zeros_like(m, dtype=np.float64)
    n = 400
    for seed in range(n):
        c, sf, s = oracle.qadamw_m_encode(m, RS, 1000 + seed)
        acc += oracle.qadamw_m_decode(c, sf, s, 16, 64, RS)
    mean = acc / n
    # one grid step of the largest block bounds the spread of a single draw
    step = 2.0 * np.float64(np.abs(_transform(m)).max()) / 4.0
    assert np.abs(mean - m).max() < 5.0 * step / np.sqrt(n)


def test_v_tile_mean_and_exact_tiles():
    rng = np.random.default_rng(9)
    # square roots on a 2^-10 grid below 4: every FP32 sum of 256 of them is exact
    r = rng.integers(1, 4096, size=(32, 64)).astype(np.float32) * np.float32(2.0 ** -10)
    r[16:, 16:32] = np.float32(0.75)  # one tile with a single BF16 value
    v = (r * r).astype(np.float32)
    codes, sf, s, mu = oracle.qadamw_v_encode(v, RS)
    exact = r.astype(np.float64).reshape(2, 16, 4, 16).mean(axis=(1, 3)).astype(np.float32)
    ref_mu = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mu, ref_mu)
    vh = oracle.qadamw_v_decode(codes, sf, s, mu, 32, 64, RS)
    assert np.array_equal(vh[16:, 16:32], v[16:, 16:32])
    assert (vh >= 0).all()
    # the square root is reconstructed within a quantisation step of the residual
    resid = r - torch.from_numpy(mu.view(np.int16)).view(torch.bfloat16).float().numpy().repeat(16, 0).repeat(16, 1)
    step = 2.0 * np.abs(resid).max()
    assert np.abs(np.sqrt(vh) - r).max() <= step


def test_v_rejects_negative_and_nonfinite():
    v = np.ones((16, 16), dtype=np.float32)
    for bad in (-1e-30, np.nan, np.inf):
        w = v.copy()
        w[3, 4] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.qadamw_v_encode(w, RS)
        assert e.value.status == oracle.ERR_NONFINITE
    with pytest.raises(oracle.OracleError) as e:
        oracle.qadamw_v_encode(np.ones((8, 16), dtype=np.float32), RS)
    assert e.value.status == oracle.ERR_UNSUPPORTED_SHAPE
