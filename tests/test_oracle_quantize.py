"""Pins for the oracle's quantiser and dequantiser (CPU only).

Invariants fixed by the format rather than by the oracle's code:
  * every dequantised value lies on {0, +-0.5, ..., +-6} x block scale x tensor scale;
  * round-to-nearest error is at most half a grid step where the block scale
    is a normal E4M3 number;
  * the block holding the tensor amax gets the largest scale (448) and the
    largest element of every normal-scaled block encodes to +-6;
  * stochastic rounding is unbiased over seeds and uses the Philox word the
    counter mapping names;
  * quantising W^T with 16x16 tiles is the transpose of quantising W.
"""
import numpy as np
import pytest

import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _codes_unpacked(codes, qk):
    lo = codes & 15
    hi = codes >> 4
    out = np.empty((codes.shape[0], qk), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def _values(codes, qk):
    c = _codes_unpacked(codes, qk)
    mag = GRID[c & 7]
    return np.where(c & 8, -mag, mag)


def _e4m3(sf):
    return np.vectorize(oracle.e4m3_value)(sf)


def _f32(x_u16):
    return (x_u16.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("block", [0, 1])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("rht", [0, 1])
def test_dequant_values_lie_on_scaled_grid(block, rounding, rht):
    x = syn.as_u16(syn.normal_with_outliers_bf16((64, 128), frac=0.01, seed=5))
    cfg = oracle.make_cfg(block=block, rounding=rounding, rht=rht, rht_seed=11, sr_seed=12)
    codes, sf, s = oracle.quantize(x, cfg)
    deq = oracle.dequantize(codes, sf, s, 64, 128)
    scale = np.repeat(_e4m3(sf), 16, axis=1) * np.float64(s)
    ratio = np.divide(deq, scale, out=np.zeros_like(deq), where=scale != 0)
    assert np.all(np.isin(np.abs(ratio), GRID))
    assert np.array_equal(deq, _values(codes, 128) * scale)


def test_rne_error_at_most_half_step():
    x = syn.as_u16(syn.normal_with_outliers_bf16((128, 256), frac=0.01, seed=6))
    codes, sf, s = oracle.quantize(x, oracle.make_cfg())
    xf = _f32(x).astype(np.float64)
    sfv = np.repeat(_e4m3(sf), 16, axis=1)
    normal = sfv >= 2.0 ** -6
    denom = (sfv.astype(np.float32) * np.float32(s)).astype(np.float64)
    v = np.abs(xf) / np.where(denom > 0, denom, 1)
    q = np.abs(_values(codes, 256))
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    step = np.where((q == 2) & (v < 2), 0.5, step)
    step = np.where((q == 4) & (v < 4), 1.0, step)
    assert np.all((np.abs(v - q) <= step / 2 + 1e-6)[normal])


def test_amax_block_gets_largest_scale_and_max_element_is_six():
    x = syn.as_u16(syn.normal_with_outliers_bf16((64, 256), frac=0.005, seed=7))
    xf = _f32(x)
    codes, sf, s = oracle.quantize(x, oracle.make_cfg())
    amax = np.abs(xf).max()
    assert s == np.float32(amax) / np.float32(2688.0)
    r, c = np.unravel_index(np.abs(xf).argmax(), xf.shape)
    assert sf[r, c // 16] == 0x7E
    u = _codes_unpacked(codes, 256)
    blocks = np.abs(xf).reshape(64, 16, 16)
    argmax = blocks.argmax(axis=2)
    for i in range(64):
        for b in range(16):
            if oracle.e4m3_value(sf[i, b]) >= 2.0 ** -6:
                assert u[i, b * 16 + argmax[i, b]] & 7 == 7


def test_zero_tensor():
    x = np.zeros((32, 64), dtype=np.uint16)
    codes, sf, s = oracle.quantize(x, oracle.make_cfg())
    assert s == 1.0 and not codes.any() and not sf.any()


def test_nonfinite_input_is_an_error():
    x = syn.as_u16(syn.normal_bf16((16, 32), seed=1)).copy()
    x[3, 5] = 0x7F80  # +inf
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize(x, oracle.make_cfg())
    assert e.value.status == oracle.ERR_NONFINITE
    x[3, 5] = 0x7FC0  # NaN
    with pytest.raises(oracle.OracleError):
        oracle.quantize(x, oracle.make_cfg())


def test_shape_rules():
    x = np.zeros((8, 24), dtype=np.uint16)
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize(x, oracle.make_cfg())
    assert e.value.status == oracle.ERR_UNSUPPORTED_SHAPE
    x = np.zeros((8, 32), dtype=np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.quantize(x, oracle.make_cfg(block=1))


def test_transpose_flag_is_a_view_change():
    x = syn.as_u16(syn.normal_bf16((48, 64), seed=8))
    a = oracle.quantize(x, oracle.make_cfg(transpose=1, rounding=1, sr_seed=3))
    b = oracle.quantize(np.ascontiguousarray(x.T), oracle.make_cfg(rounding=1, sr_seed=3))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_16x16_quantisation_commutes_with_transpose():
    w = syn.as_u16(syn.normal_with_outliers_bf16((64, 96), frac=0.01, seed=9))
    c1, sf1, s1 = oracle.quantize(w, oracle.make_cfg(block=1))
    c2, sf2, s2 = oracle.quantize(w, oracle.make_cfg(block=1, transpose=1))
    assert s1 == s2
    assert np.array_equal(_codes_unpacked(c1, 96).T, _codes_unpacked(c2, 64))
    assert np.array_equal(sf1[::16, :].T, sf2[::16, :])


def test_16x16_scale_is_shared_by_the_tile():
    w = syn.as_u16(syn.normal_bf16((32, 64), seed=10))
    _, sf, s = oracle.quantize(w, oracle.make_cfg(block=1))
    for t in range(2):
        assert np.all(sf[16 * t:16 * t + 16] == sf[16 * t])
    wf = np.abs(_f32(w))
    tmax = wf.reshape(2, 16, 4, 16).max(axis=(1, 3))
    expect = [[oracle.e4m3_encode(np.float32(np.float32(tmax[i, j]) / np.float32(6.0)) / s)
               for j in range(4)] for i in range(2)]
    assert np.array_equal(sf[::16], np.array(expect, dtype=np.uint8))


def test_sr_uses_the_named_philox_word():
    # Blocks of 0.25 with one 6.0 per block: the scaled elements sit at (or
    # within an ulp of) the midpoint f = 1/2 between grid points 0 and 0.5, so
    # each one rounds up or down according to its own Philox word.
    qk = 64
    x = np.full((4, qk), 0x3E80, dtype=np.uint16)  # 0.25
    x[:, 0::16] = 0x40C0                           # 6.0 -> block scale 1.0 after rounding
    seed, offset = 0x0123456789ABCDEF, 0x42
    codes, sf, s = oracle.quantize(x, oracle.make_cfg(rounding=1, sr_seed=seed, sr_offset=offset))
    assert np.all(sf == 0x7E)
    denom = np.float32(np.float32(oracle.e4m3_value(sf[0, 0])) * s)
    v = np.float32(np.float32(0.25) / denom)
    ups = 0
    u = _codes_unpacked(codes, qk)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in range(4):
        for k in range(qk):
            if k % 16 == 0:
                continue
            e = i * qk + k
            w = oracle.philox4x32_10([e >> 2, e >> 34, offset & 0xFFFFFFFF, offset >> 32], key)[e & 3]
            lo_code = int(np.searchsorted(GRID, v, side="right") - 1)
            f = (v - GRID[lo_code]) / (GRID[lo_code + 1] - GRID[lo_code])
            up = (int(w) >> 8) * 2.0 ** -24 < f
            assert u[i, k] == lo_code + (1 if up else 0), (i, k)
            ups += up
    assert 0 < ups < 4 * 60


def test_sr_is_unbiased_over_seeds():
    x = syn.as_u16(syn.normal_bf16((2, 32), seed=11))
    acc = np.zeros((2, 32))
    n = 2000
    ref = None
    for seed in range(n):
        codes, sf, s = oracle.quantize(x, oracle.make_cfg(rounding=1, sr_seed=seed))
        d = oracle.dequantize(codes, sf, s, 2, 32)
        acc += d
        if ref is None:
            ref = (sf, s)
        assert np.array_equal(sf, ref[0])  # the scales do not depend on the draws
    mean = acc / n
    xf = _f32(x).astype(np.float64)
    scale = np.repeat(_e4m3(ref[0]), 16, axis=1) * ref[1]
    sigma = scale * 2.0 * 0.5 / np.sqrt(n)
    # elements whose scaled magnitude exceeds 6 saturate (a property of the
    # format, not of the rounding); every other element is unbiased
    inside = np.abs(xf) / scale < 6.0
    assert inside.sum() >= 60
    assert np.all((np.abs(mean - xf) < 4 * sigma + 1e-12)[inside])


def test_rht_quantisation_roundtrip_is_close():
    x = syn.as_u16(syn.normal_bf16((16, 128), seed=12))
    cfg = oracle.make_cfg(rht=1, rht_seed=77)
    codes, sf, s = oracle.quantize(x, cfg)
    d = oracle.dequantize(codes, sf, s, 16, 128).astype(np.float32)
    sigma = oracle.rht_signs(77)
    back = np.stack([np.concatenate([oracle.rht16(d[i, k:k + 16], np.ones(16, np.float32)) * sigma
                                     for k in range(0, 128, 16)]) for i in range(16)])
    xf = _f32(x)
    rel = np.linalg.norm(back - xf) / np.linalg.norm(xf)
    assert rel < 0.15
    # amax is taken after the transform
    assert s == np.float32(oracle.amax(x, cfg)) / np.float32(2688.0)
    assert oracle.amax(x, cfg) != np.abs(xf).max()


def test_sf_mma_layout_positions():
    qk = 256  # 16 scales per row -> 4 K atoms
    assert oracle.sf_mma_offset(0, 0, qk) == 0
    assert oracle.sf_mma_offset(0, 1, qk) == 1
    assert oracle.sf_mma_offset(0, 3, qk) == 3
    assert oracle.sf_mma_offset(1, 0, qk) == 16
    assert oracle.sf_mma_offset(31, 0, qk) == 31 * 16
    assert oracle.sf_mma_offset(32, 0, qk) == 4
    assert oracle.sf_mma_offset(127, 3, qk) == 31 * 16 + 3 * 4 + 3
    assert oracle.sf_mma_offset(0, 4, qk) == 512
    assert oracle.sf_mma_offset(128, 0, qk) == 4 * 512
    # bijective on the padded layout
    qr = 256
    offs = sorted(oracle.sf_mma_offset(r, kb, qk) for r in range(qr) for kb in range(qk // 16))
    assert offs == list(range(oracle.sf_mma_bytes(qr, qk)))
    # padding: 100 rows x 20 scales -> 1 row atom x 5 K atoms; unused bytes stay zero
    sf = np.arange(1, 100 * 20 + 1, dtype=np.int64).astype(np.uint8).reshape(100, 20)
    sf[sf == 0] = 1
    mma = oracle.sf_to_mma(sf, 100, 320)
    assert mma.size == 5 * 512
    assert np.count_nonzero(mma) == 100 * 20
