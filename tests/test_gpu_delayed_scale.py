"""Delayed scaling on the GPU: nvfp4_quantize_given_amax against the oracle's
quantize_given_amax (bit-exact codes, block scales and tensor scale), and
nvfp4_gemm_quantize, the GEMM whose epilogue quantises D for the next layer.

The fused epilogue is checked three ways:
  * hand-built unit-scale operands make D exact, so the oracle's FP64 GEMM,
    rounded to BF16, is the fused kernel's D bit for bit, and the oracle's
    delayed-scaling quantisation of it must equal the fused codes and scales;
  * on quantised random operands the fused kernel's D equals nvfp4_gemm's D
    and its codes equal nvfp4_quantize_given_amax applied to that D;
  * edge cases: ragged M, N, K, single-CTA and pair modes, both scale layouts,
    no D store, bad amax, empty shapes.
"""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import ALL_MODES, DEV, assert_quant_equal, cfgs, mode_id

pytestmark = pytest.mark.gpu


def _amax_dev(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def _f32(x_u16):
    return (x_u16.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ quantiser
@pytest.mark.parametrize("mode", ALL_MODES, ids=mode_id)
@pytest.mark.parametrize("transpose", [0, 1])
@pytest.mark.parametrize("factor", [1.0, 2.5, 0.2])
def test_given_amax_matches_oracle(mode, transpose, factor):
    x = syn.normal_with_outliers_bf16((144, 272), frac=0.01, seed=61)
    g, o = cfgs(transpose=transpose, **mode)
    qr = 272 if transpose else 144
    if mode["block"] == 1 and qr % 16:
        pytest.skip("16x16 blocks need qr % 16 == 0")
    own = oracle.amax(syn.as_u16(x), o)
    amax = np.float32(own * factor)
    q = nv.nvfp4_quantize_given_amax(x.to(DEV), g, _amax_dev(amax))
    assert_quant_equal(q, oracle.quantize_given_amax(syn.as_u16(x), o, amax))


def test_given_own_amax_equals_two_pass_quantiser():
    x = syn.normal_with_outliers_bf16((384, 640), frac=0.01, seed=62)
    g, o = cfgs()
    amax = oracle.amax(syn.as_u16(x), o)
    a = nv.nvfp4_quantize(x.to(DEV), g)
    b = nv.nvfp4_quantize_given_amax(x.to(DEV), g, _amax_dev(amax))
    assert torch.equal(a.codes, b.codes) and torch.equal(a.sf, b.sf) and torch.equal(a.tensor_scale, b.tensor_scale)


def test_given_amax_rowmajor_ragged_and_zero():
    x = syn.normal_bf16((200, 336), seed=63)
    g, o = cfgs(sf_layout=nv.NVFP4_SF_ROWMAJOR)
    for amax in (np.float32(0.0), np.float32(1.7)):
        q = nv.nvfp4_quantize_given_amax(x.to(DEV), g, _amax_dev(amax))
        assert_quant_equal(q, oracle.quantize_given_amax(syn.as_u16(x), o, amax))


def test_given_amax_bad_amax_and_nonfinite_input():
    x = syn.normal_bf16((64, 128), seed=64)
    g, _ = cfgs()
    for bad in (float("nan"), float("inf"), -2.0):
        ws = torch.zeros(nv.nvfp4_quantize_workspace_size(64, 128, g), dtype=torch.uint8, device=DEV)
        q = nv.nvfp4_quantize_given_amax(x.to(DEV), g, _amax_dev(bad), workspace=ws)
        assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_NONFINITE
        assert torch.isnan(q.tensor_scale).all()
    y = x.clone()
    y[5, 17] = float("inf")
    ws = torch.zeros(nv.nvfp4_quantize_workspace_size(64, 128, g), dtype=torch.uint8, device=DEV)
    nv.nvfp4_quantize_given_amax(y.to(DEV), g, _amax_dev(3.0), workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_NONFINITE
    # and the workspace is clean again for a finite input
    nv.nvfp4_quantize_given_amax(x.to(DEV), g, _amax_dev(3.0), workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK


# ------------------------------------------------------ fused GEMM epilogue
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _pack(c4):
    return (c4[:, 0::2] | (c4[:, 1::2] << 4)).astype(np.uint8)


def _unit_operand(rng, rows, k):
    c4 = rng.integers(0, 16, size=(rows, k), dtype=np.uint8)
    codes = _pack(c4)
    sf = np.full((rows, k // 16), 0x38, dtype=np.uint8)  # E4M3 1.0
    t = nv.NVFP4Tensor(codes=torch.from_numpy(codes).to(DEV),
                       sf=torch.from_numpy(oracle.sf_to_mma(sf, rows, k)).to(DEV),
                       tensor_scale=torch.ones(1, dtype=torch.float32, device=DEV),
                       rows=rows, k=k, sf_layout=nv.NVFP4_SF_MMA)
    return t, (codes, sf, np.float32(1.0))


def _bf16_bits(d64):
    # exact FP64 sums that fit FP32 -> FP32 (exact) -> BF16 round to nearest even
    t = torch.from_numpy(d64.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (200, 96, 96), (72, 160, 320),
                                   (384, 288, 1024), (1, 32, 32)])
@pytest.mark.parametrize("sf_layout", [nv.NVFP4_SF_MMA, nv.NVFP4_SF_ROWMAJOR], ids=["mma", "rowmajor"])
@pytest.mark.parametrize("amax_kind", ["exact", "double", "half", "zero"])
def test_fused_exact_operands_match_oracle(M, N, K, sf_layout, amax_kind):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a, oa = _unit_operand(rng, M, K)
    b, ob = _unit_operand(rng, N, K)
    y = _bf16_bits(oracle.gemm_f64(oa, ob, M, N, K))
    own = np.float32(np.abs(_f32(y)).max())
    amax = {"exact": own, "double": own * np.float32(2), "half": own * np.float32(0.5), "zero": np.float32(0)}[amax_kind]
    amax_out = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    d, q = nv.nvfp4_gemm_quantize(a, b, _amax_dev(amax), sf_layout=sf_layout, amax_out=amax_out)
    got_d = d.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_d, y), "fused D differs from the exact product rounded to BF16"
    assert amax_out.item() == own
    _, o = cfgs(sf_layout=sf_layout)
    assert_quant_equal(q, oracle.quantize_given_amax(y, o, amax))


def _quantised(x, **mode):
    g, _ = cfgs(**mode)
    return nv.nvfp4_quantize(x.to(DEV), g)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (640, 384, 768), (1000, 544, 1056), (128, 1024, 512),
                                   (96, 64, 64)])
@pytest.mark.parametrize("sf_layout", [nv.NVFP4_SF_MMA, nv.NVFP4_SF_ROWMAJOR], ids=["mma", "rowmajor"])
def test_fused_equals_gemm_then_given_amax_quantiser(M, N, K, sf_layout):
    x = syn.normal_with_outliers_bf16((M, K), frac=0.01, seed=M + K)
    w = syn.normal_bf16((N, K), seed=N + K, std=0.02)
    qa, qb = _quantised(x), _quantised(w, block=1)
    d_plain = nv.nvfp4_gemm(qa, qb)
    amax = _amax_dev(float(d_plain.abs().max().float()) * 0.9)
    amax_out = torch.zeros(1, dtype=torch.float32, device=DEV)
    d, q = nv.nvfp4_gemm_quantize(qa, qb, amax, sf_layout=sf_layout, amax_out=amax_out)
    assert torch.equal(d, d_plain)
    assert amax_out.item() == d_plain.abs().max().float().item()
    g, _ = cfgs(sf_layout=sf_layout)
    ref = nv.nvfp4_quantize_given_amax(d_plain, g, amax)
    assert torch.equal(q.tensor_scale, ref.tensor_scale)
    assert torch.equal(q.codes, ref.codes)
    assert torch.equal(q.sf, ref.sf)


def test_fused_without_d_store_and_reuse():
    x = syn.normal_bf16((512, 256), seed=71)
    w = syn.normal_bf16((256, 256), seed=72, std=0.02)
    qa, qb = _quantised(x), _quantised(w, block=1)
    amax = _amax_dev(0.05)
    d, q1 = nv.nvfp4_gemm_quantize(qa, qb, amax)
    none, q2 = nv.nvfp4_gemm_quantize(qa, qb, amax, store_d=False)
    assert none is None
    assert torch.equal(q1.codes, q2.codes) and torch.equal(q1.sf, q2.sf)


def test_fused_bad_amax_reports_and_keeps_d():
    x = syn.normal_bf16((256, 256), seed=73)
    w = syn.normal_bf16((256, 256), seed=74, std=0.02)
    qa, qb = _quantised(x), _quantised(w, block=1)
    d_plain = nv.nvfp4_gemm(qa, qb)
    for bad in (float("nan"), float("-inf"), -1.0):
        ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
        d, q = nv.nvfp4_gemm_quantize(qa, qb, _amax_dev(bad), workspace=ws)
        assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_NONFINITE
        assert torch.isnan(q.tensor_scale).all()
        assert torch.equal(d, d_plain)


def test_fused_shape_rules_and_empty():
    x = syn.normal_bf16((128, 64), seed=75)
    qa = _quantised(x)
    qb = _quantised(syn.normal_bf16((48, 64), seed=76))  # N = 48: not a multiple of 32
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_gemm_quantize(qa, qb, _amax_dev(1.0))
    assert e.value.status == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    empty = _quantised(torch.zeros((0, 64), dtype=torch.bfloat16))
    qb2 = _quantised(syn.normal_bf16((64, 64), seed=77))
    d, q = nv.nvfp4_gemm_quantize(empty, qb2, _amax_dev(1.0))
    torch.cuda.synchronize()
    assert d.shape == (0, 64) and q.codes.shape == (0, 32)


def test_fused_full_size_fprop():
    # the MLP up-projection fprop: Y [8192, 20480] quantised for the next
    # layer with last step's amax (here: this step's, times 1.1)
    x, w, _ = syn.config2()
    gx, _ = cfgs()
    gw, _ = cfgs(block=1)
    qa = nv.nvfp4_quantize(x.to(DEV), gx)
    qb = nv.nvfp4_quantize(w.to(DEV), gw)
    d_plain = nv.nvfp4_gemm(qa, qb)
    amax = _amax_dev(float(d_plain.abs().max().float()) * 1.1)
    amax_out = torch.zeros(1, dtype=torch.float32, device=DEV)
    d, q = nv.nvfp4_gemm_quantize(qa, qb, amax, amax_out=amax_out)
    assert torch.equal(d, d_plain)
    ref = nv.nvfp4_quantize_given_amax(d_plain, gx, amax)
    assert torch.equal(q.codes, ref.codes) and torch.equal(q.sf, ref.sf)
    assert torch.equal(q.tensor_scale, ref.tensor_scale)
    assert amax_out.item() == d_plain.abs().max().float().item()
