"""Pins for the oracle's codecs and random stream (CPU only).

Each check compares the oracle with something fixed outside it: the E2M1
grid and tie table of the format, torch's float8_e4m3fn conversion, a
brute-force nearest search written here in numpy, and the published
Philox4x32-10 known-answer vectors.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e2m1_grid_matches_format():
    rows = [r for r in _read_golden("e2m1_grid.txt") if r[0] == "grid"]
    for _, code, value in rows:
        assert oracle.e2m1_value(int(code)) == float(value)
        assert oracle.e2m1_value(int(code) | 8) == -float(value)


def test_e2m1_rne_tie_table():
    rows = [r for r in _read_golden("e2m1_grid.txt") if r[0] == "tie"]
    assert len(rows) == 7
    for _, v, code in rows:
        assert oracle.e2m1_encode_rne(float(v)) == int(code), v
        assert oracle.e2m1_encode_rne(-float(v)) == int(code) | 8, v


def _brute_nearest_even(v):
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    d = np.abs(grid - abs(v))
    best = np.flatnonzero(d == d.min())
    code = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
    return int(code) | (8 if np.signbit(v) else 0)


def test_e2m1_rne_brute_force():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.uniform(-8, 8, 20000).astype(np.float32),
        np.float32([0.0, -0.0, 6.0, 7.0, 100.0, -100.0, 1e-30, -1e-30]),
        # one float step either side of every midpoint
        np.nextafter(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), np.float32(0)),
        np.nextafter(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), np.float32(10)),
    ])
    for v in vals:
        assert oracle.e2m1_encode_rne(v) == _brute_nearest_even(v), v


def test_e2m1_negative_zero_keeps_sign():
    assert oracle.e2m1_encode_rne(-0.1) == 0x8
    assert oracle.e2m1_encode_rne(-0.0) == 0x8
    assert oracle.e2m1_encode_rne(0.0) == 0x0


def test_e4m3_decode_all_bytes_match_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for byte in range(256):
        got = oracle.e4m3_value(byte)
        if np.isnan(ref[byte]):
            assert np.isnan(got), byte
        else:
            assert got == ref[byte], byte
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(2)
    finite = np.array([oracle.e4m3_value(b) for b in range(127)], dtype=np.float32)
    mids = ((finite[:-1].astype(np.float64) + finite[1:]) / 2).astype(np.float32)
    samples = np.concatenate([
        finite, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
        np.exp(rng.uniform(np.log(1e-5), np.log(464.0), 20000)).astype(np.float32),
        np.float32([0.0, 2.0 ** -10, 3 * 2.0 ** -11, 464.0]),
    ])
    samples = samples[samples <= 464.0]
    ref = torch.from_numpy(samples).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t, r in zip(samples, ref):
        assert oracle.e4m3_encode(t) == r, t


def test_e4m3_encode_saturates():
    for t in [448.0, 460.0, 464.0, 465.0, 479.0, 500.0, 1e6, 3.0e38]:
        assert oracle.e4m3_encode(t) == 0x7E, t


def test_e4m3_roundtrip_identity():
    for b in range(127):
        assert oracle.e4m3_encode(oracle.e4m3_value(b)) == b


def test_philox_known_answers():
    rows = _read_golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        out = oracle.philox4x32_10(vals[0:4], vals[4:6])
        assert list(out) == vals[6:10]


def test_philox_uniformity():
    # 4096 draws of 4 words: the top byte of each word is near-uniform.
    words = np.concatenate([oracle.philox4x32_10([i, 0, 7, 0], [123, 456]) for i in range(4096)])
    hist = np.bincount(words >> 24, minlength=256)
    expected = words.size / 256
    chi2 = ((hist - expected) ** 2 / expected).sum()
    assert chi2 < 256 + 6 * np.sqrt(2 * 256)


@pytest.mark.parametrize("lo,hi", [(0.0, 0.5), (0.5, 1.0), (1.0, 1.5), (1.5, 2.0), (2.0, 3.0), (3.0, 4.0), (4.0, 6.0)])
def test_e2m1_sr_stays_on_bracket_and_is_unbiased(lo, hi):
    rng = np.random.default_rng(3)
    grid = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}
    for v in np.float32([lo + (hi - lo) * f for f in (0.1, 0.37, 0.5, 0.9)]):
        draws = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64)
        vals = np.array([grid[oracle.e2m1_encode_sr(v, int(r))] for r in draws])
        assert set(np.unique(vals)) <= {lo, hi}
        sigma = (hi - lo) * 0.5 / np.sqrt(len(vals))
        assert abs(vals.mean() - v) < 4 * sigma + 1e-9
        # the sign is carried like round-to-nearest
        assert oracle.e2m1_encode_sr(-v, int(draws[0])) & 8


def test_e2m1_sr_threshold_rule():
    # u = (r >> 8) * 2^-24; round up iff u < f.  At f = 0.5 that is r < 2^31.
    assert oracle.e2m1_encode_sr(0.25, 0x7FFFFFFF) == 1
    assert oracle.e2m1_encode_sr(0.25, 0x80000000) == 0
    # on a grid point f = 0: never rounds up, whatever the draw
    for r in (0, 1, 0xFFFFFFFF):
        assert oracle.e2m1_encode_sr(1.5, r) == 3
    assert oracle.e2m1_encode_sr(7.0, 0) == 7
