"""Quantised AdamW state codec on the GPU against the oracle: codes, block
scales, tensor scales and tile means bit for bit, decoded states bit for bit
(the decoders are fixed sequences of FP32 operations), on ragged shapes, heavy
tails, zero tensors and an optimizer-state-sized tensor; bad inputs reported."""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle

from _helpers import DEV

pytestmark = pytest.mark.gpu

RS, SS, SO = 0x5EED, 0xBEEF, 3


def _m(rows, cols, seed, scale=1e-3):
    g = torch.Generator().manual_seed(seed)
    m = torch.randn((rows, cols), generator=g) * scale
    m[:: 7, :: 13] *= 40.0  # heavy tail
    return m


def _v(rows, cols, seed, scale=1e-3):
    g = torch.Generator().manual_seed(seed)
    v = (torch.randn((rows, cols), generator=g) * scale) ** 2
    v *= torch.exp(torch.randn((rows, 1), generator=g))  # row-dependent magnitude
    return v


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("shape", [(16, 16), (48, 128), (37, 272), (300, 4112)], ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("scale", [1e-4, 1.0])
def test_m_encode_decode_match_oracle(shape, scale):
    rows, cols = shape
    m = _m(rows, cols, seed=rows + cols, scale=scale)
    st = nv.nvfp4_qadamw_m_encode(m.to(DEV), RS, SS, SO)
    codes, sf, s = oracle.qadamw_m_encode(m.numpy(), RS, SS, SO)
    assert st.tensor_scale.item() == s
    assert np.array_equal(st.sf.cpu().numpy(), sf)
    assert np.array_equal(st.codes.cpu().numpy(), codes)
    got = nv.nvfp4_qadamw_m_decode(st, RS)
    ref = oracle.qadamw_m_decode(codes, sf, s, rows, cols, RS)
    assert np.array_equal(_bits(got), ref.view(np.uint32))


@pytest.mark.parametrize("shape", [(16, 16), (48, 128), (64, 272), (320, 4112)], ids=lambda s: "%dx%d" % s)
def test_v_encode_decode_match_oracle(shape):
    rows, cols = shape
    v = _v(rows, cols, seed=rows * 3 + cols)
    st = nv.nvfp4_qadamw_v_encode(v.to(DEV), RS)
    codes, sf, s, mu = oracle.qadamw_v_encode(v.numpy(), RS)
    assert st.tensor_scale.item() == s
    assert np.array_equal(st.tile_mean.cpu().numpy().view(np.uint16), mu)
    assert np.array_equal(st.sf.cpu().numpy(), sf)
    assert np.array_equal(st.codes.cpu().numpy(), codes)
    got = nv.nvfp4_qadamw_v_decode(st, RS)
    ref = oracle.qadamw_v_decode(codes, sf, s, mu, rows, cols, RS)
    assert np.array_equal(_bits(got), ref.view(np.uint32))


def test_zero_states():
    z = torch.zeros((32, 64))
    st = nv.nvfp4_qadamw_m_encode(z.to(DEV), RS, SS)
    assert st.tensor_scale.item() == 1.0 and not st.codes.any() and not st.sf.any()
    assert not nv.nvfp4_qadamw_m_decode(st, RS).any()
    sv = nv.nvfp4_qadamw_v_encode(z.to(DEV), RS)
    assert not sv.tile_mean.any() and not nv.nvfp4_qadamw_v_decode(sv, RS).any()


def test_v_bad_values_and_shapes():
    v = _v(32, 64, seed=5)
    for bad in (-1.0, float("nan"), float("inf")):
        w = v.clone()
        w[3, 9] = bad
        ws = torch.zeros(nv.nvfp4_qadamw_workspace_size(), dtype=torch.uint8, device=DEV)
        st = nv.nvfp4_qadamw_v_encode(w.to(DEV), RS, workspace=ws)
        assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_NONFINITE
        assert torch.isnan(st.tensor_scale).all()
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_qadamw_v_encode(torch.ones((24, 64), device=DEV), RS)
    assert e.value.status == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_qadamw_m_encode(torch.ones((24, 40), device=DEV), RS, SS)
    assert e.value.status == nv.NVFP4_ERR_UNSUPPORTED_SHAPE


def test_large_state_matches_oracle():
    # a 2048 x 5120 moment (10.5 M elements), compared whole
    rows, cols = 2048, 5120
    m = _m(rows, cols, seed=21)
    st = nv.nvfp4_qadamw_m_encode(m.to(DEV), RS, SS)
    codes, sf, s = oracle.qadamw_m_encode(m.numpy(), RS, SS)
    assert st.tensor_scale.item() == s
    assert np.array_equal(st.sf.cpu().numpy(), sf) and np.array_equal(st.codes.cpu().numpy(), codes)
    v = _v(rows, cols, seed=22)
    sv = nv.nvfp4_qadamw_v_encode(v.to(DEV), RS)
    codes, sf, s, mu = oracle.qadamw_v_encode(v.numpy(), RS)
    assert sv.tensor_scale.item() == s
    assert np.array_equal(sv.tile_mean.cpu().numpy().view(np.uint16), mu)
    assert np.array_equal(sv.sf.cpu().numpy(), sf) and np.array_equal(sv.codes.cpu().numpy(), codes)


def test_weight_sized_states_properties():
    # moments of the 20480 x 5120 up-projection weight: decoded states close
    # to the input.  The oracle on 2048 x 5120 of the same recipe stays below
    # 0.52 x the run's largest magnitude (first moment) and 0.19 x the tile's
    # spread plus its mean's BF16 rounding (second moment); the bounds below
    # (2 and 1) leave room for the larger tensor and catch layout errors.
    rows, cols = 20480, 5120
    m = _m(rows, cols, seed=11)
    st = nv.nvfp4_qadamw_m_encode(m.to(DEV), RS, SS)
    mh = nv.nvfp4_qadamw_m_decode(st, RS).cpu()
    blk = m.abs().reshape(rows, cols // 16, 16).amax(dim=2).repeat_interleave(16, dim=1)
    assert bool(((mh - m).abs() <= 2.0 * blk).all())
    v = _v(rows, cols, seed=12)
    sv = nv.nvfp4_qadamw_v_encode(v.to(DEV), RS)
    vh = nv.nvfp4_qadamw_v_decode(sv, RS).cpu()
    assert bool((vh >= 0).all())
    r = v.sqrt()
    tile = r.reshape(rows // 16, 16, cols // 16, 16)
    hi, lo = tile.amax(dim=(1, 3)), tile.amin(dim=(1, 3))
    # residual bound: the tile's spread plus the BF16 rounding of its mean
    bound = (hi - lo + hi * 2.0 ** -8).repeat_interleave(16, 0).repeat_interleave(16, 1)
    assert bool(((vh.sqrt() - r).abs() <= 1.0 * bound).all())
