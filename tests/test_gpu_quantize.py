"""GPU quantiser parity with the oracle: codes, block-scale bytes and the
tensor scale must match bit for bit, for every mode, orientation and scale
layout, on small ragged shapes, on hand-built edge cases and on sampled rows
of the full-size quantise sweep."""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import ALL_MODES, DEV, assert_quant_equal, cfgs, mode_id, quant_pair

pytestmark = pytest.mark.gpu

SMALL = [(16, 16), (64, 256), (48, 160), (256, 256), (33, 4096), (130, 528), (1024, 1024)]


@pytest.mark.parametrize("mode", ALL_MODES, ids=mode_id)
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("layout", [nv.NVFP4_SF_MMA, nv.NVFP4_SF_ROWMAJOR], ids=["mma", "rowmajor"])
def test_rowwise_parity(mode, shape, layout):
    if mode["block"] == 1 and shape[0] % 16:
        pytest.skip("16x16 blocks need rows % 16 == 0")
    x = syn.normal_with_outliers_bf16(shape, frac=0.01, seed=shape[0] * 131 + shape[1])
    q, o = quant_pair(x, sf_layout=layout, **mode)
    assert_quant_equal(q, o)


@pytest.mark.parametrize("mode", ALL_MODES, ids=mode_id)
@pytest.mark.parametrize("shape", [(16, 16), (256, 64), (160, 48), (160, 56), (512, 136), (4096, 40)],
                         ids=lambda s: "%dx%d" % s)
def test_transposed_parity(mode, shape):
    if mode["block"] == 1 and shape[1] % 16:
        pytest.skip("16x16 blocks need cols % 16 == 0 when transposed")
    x = syn.normal_with_outliers_bf16(shape, frac=0.01, seed=shape[0] * 7 + shape[1])
    q, o = quant_pair(x, transpose=1, **mode)
    assert_quant_equal(q, o)


def test_strided_input():
    base = syn.normal_bf16((64, 320), seed=3)
    view = base.to(DEV)[:, 32:288]  # row stride 320, 256 columns
    g, o = cfgs()
    q = nv.nvfp4_quantize(view, g)
    ref = oracle.quantize(syn.as_u16(base[:, 32:288].contiguous()), o)
    assert_quant_equal(q, ref)


def _edge_tensor():
    # amax = 10.5 makes the tensor scale s = 10.5 / 2688 = 2^-8 exactly; a
    # block led by 10.5 then gets block scale 448 and divisor d = 1.75, so
    # x = m * 1.75 (exact in BF16) lands exactly on the E2M1 midpoint m.  The
    # rest probe zeros of both signs, values that round to (negative) zero,
    # saturation, a block whose scale rounds to zero, and an ordinary block.
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for sgn in (1.0, -1.0):
        rows.append([10.5] + [sgn * m * 1.75 for m in mids]
                    + [sgn * 0.0, sgn * 1e-30, sgn * 0.1, sgn * 0.2, sgn * 10.4, sgn * 10.5, sgn * 0.42, sgn * 7.0])
    rows.append([1e-8, -1e-8] * 8)
    rows.append([1.0, -0.3, 0.7, 0.05, -0.9, 0.33, 0.1, -0.6, 0.8, 0.2, -0.44, 0.5, 0.01, -1.0, 0.77, 0.25])
    x = torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)
    return x.repeat(4, 1)  # 16 rows


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("block", [0, 1])
def test_edge_values(rounding, block):
    x = _edge_tensor()
    q, o = quant_pair(x, block=block, rounding=rounding)
    assert o[2] == np.float32(2.0 ** -8)
    assert_quant_equal(q, o)


def test_zero_tensor():
    x = torch.zeros((32, 64), dtype=torch.bfloat16)
    q, o = quant_pair(x)
    assert_quant_equal(q, o)
    assert q.tensor_scale.item() == 1.0


def test_nonfinite_sets_status():
    x = syn.normal_bf16((32, 64), seed=1)
    x[5, 7] = float("inf")
    g, _ = cfgs()
    ws = torch.zeros(nv.nvfp4_quantize_workspace_size(32, 64, g), dtype=torch.uint8, device=DEV)
    q = nv.nvfp4_quantize(x.to(DEV), g, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_NONFINITE
    assert np.isnan(q.tensor_scale.item())
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK  # cleared
    x[5, 7] = float("nan")
    nv.nvfp4_quantize(x.to(DEV), g, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_NONFINITE
    # the workspace is usable again afterwards
    x[5, 7] = 1.0
    q = nv.nvfp4_quantize(x.to(DEV), g, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
    assert np.isfinite(q.tensor_scale.item())


def test_empty_tensor():
    g, _ = cfgs()
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    q = nv.nvfp4_quantize(x, g)
    torch.cuda.synchronize()
    assert q.tensor_scale.item() == 1.0


def test_deterministic_and_seed_sensitive():
    x = syn.normal_bf16((128, 512), seed=4).to(DEV)
    g1, _ = cfgs(rounding=1, rht=1, sr_seed=1)
    g2, _ = cfgs(rounding=1, rht=1, sr_seed=2)
    a = nv.nvfp4_quantize(x, g1).codes
    b = nv.nvfp4_quantize(x, g1).codes
    c = nv.nvfp4_quantize(x, g2).codes
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


# ---- full-size quantise sweep (sampled rows, same launch configuration) ----
@pytest.mark.parametrize("mode", ALL_MODES, ids=mode_id)
@pytest.mark.parametrize("shape_idx", [0, 1], ids=["4096x5120", "8192x20480"])
def test_sweep_full_size_sampled(mode, shape_idx):
    x = syn.config1(shape_idx)
    g, o = cfgs(**mode)
    q = nv.nvfp4_quantize(x.to(DEV), g)
    qr = x.shape[0]
    # whole 16-row groups so that 16x16 tiles are complete: first, one in the
    # middle, last
    rng = np.random.default_rng(shape_idx)
    groups = [0, int(rng.integers(1, qr // 16 - 1)), qr // 16 - 1]
    xs = syn.as_u16(x)
    for gidx in groups:
        r0 = int(gidx) * 16
        ref = oracle.quantize_rows(xs, o, r0, r0 + 16)
        assert_quant_equal(q, ref, rows=np.arange(r0, r0 + 16))


@pytest.mark.parametrize("pass_", [1, 2], ids=["amax-pass", "encode-pass"])
def test_quantize_timeout_is_reported_and_context_survives(pass_):
    x = syn.normal_bf16((512, 1024), seed=41)
    g, o = cfgs(rounding=1, rht=1)
    ws = torch.zeros(nv.nvfp4_quantize_workspace_size(512, 1024, g), dtype=torch.uint8, device=DEV)
    xd = x.to(DEV)
    nv.nvfp4_debug_quantize_skip_load(pass_)
    q = nv.nvfp4_quantize(xd, g, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_TIMEOUT
    assert np.isnan(q.tensor_scale.cpu().numpy()[0])
    # one-shot hook; the context is still usable and the next call is exact
    q = nv.nvfp4_quantize(xd, g, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
    assert_quant_equal(q, oracle.quantize(syn.as_u16(x), o))
