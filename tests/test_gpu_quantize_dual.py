"""nvfp4_quantize_dual: both outputs of one read must equal the oracle's
quantisation with each output's own configuration, bit for bit, and equal
what nvfp4_quantize produces for that configuration alone.  Also covers the
quantiser's extreme ranges (tensor scales far from 1, tiny elements next to
huge ones), where the element division leaves its fast path."""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import DEV, assert_quant_equal, cfgs

pytestmark = pytest.mark.gpu

S = nv.NVFP4_DEFAULT_RHT_SEED

# (output A, output B) as used by a training step, plus mixed cases.
PAIRS = {
    "act-row-rne+col-sr-rht": (dict(), dict(transpose=1, rounding=1, rht=1, rht_seed=S, sr_seed=5)),
    "weight-16x16-both": (dict(block=1), dict(block=1, transpose=1)),
    # the transposed output listed first, and mixed scale layouts: the kernel
    # copies the transposed codes from the row output's tile either way
    "weight-16x16-col-first": (dict(block=1, transpose=1), dict(block=1)),
    "weight-16x16-mixed-sf": (dict(block=1, sf_layout=nv.NVFP4_SF_ROWMAJOR), dict(block=1, transpose=1)),
    "row-rne+col-rne": (dict(), dict(transpose=1)),
    "row-sr-rht+col-sr-rht": (dict(rounding=1, rht=1, sr_seed=9), dict(transpose=1, rounding=1, rht=1, sr_seed=10)),
    "col-16x16-sr+row-rht": (dict(block=1, transpose=1, rounding=1), dict(rht=1)),
    "row+row-sr": (dict(), dict(rounding=1, sr_seed=3)),
}

SHAPES = [(16, 16), (128, 128), (144, 272), (256, 640), (400, 96), (1040, 1312)]


def _oracle(x_cpu, mode):
    return oracle.quantize(syn.as_u16(x_cpu), cfgs(**mode)[1])


@pytest.mark.parametrize("pair", list(PAIRS), ids=list(PAIRS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
def test_dual_matches_oracle(pair, shape):
    ma, mb = PAIRS[pair]
    for m in (ma, mb):
        qr = shape[1] if m.get("transpose") else shape[0]
        if m.get("block") == 1 and qr % 16:
            pytest.skip("16x16 blocks need qr % 16 == 0")
    x = syn.normal_with_outliers_bf16(shape, frac=0.01, seed=shape[0] * 17 + shape[1])
    ga, gb = cfgs(**ma)[0], cfgs(**mb)[0]
    qa, qb = nv.nvfp4_quantize_dual(x.to(DEV), ga, gb)
    assert_quant_equal(qa, _oracle(x, ma))
    assert_quant_equal(qb, _oracle(x, mb))
    # the same outputs as two single-output calls
    sa = nv.nvfp4_quantize(x.to(DEV), ga)
    sb = nv.nvfp4_quantize(x.to(DEV), gb)
    for d, s in ((qa, sa), (qb, sb)):
        assert torch.equal(d.codes, s.codes)
        assert torch.equal(d.sf, s.sf)
        assert torch.equal(d.tensor_scale, s.tensor_scale)


def test_dual_rowmajor_scales():
    x = syn.normal_bf16((272, 208), seed=44)
    ma = dict(sf_layout=nv.NVFP4_SF_ROWMAJOR)
    mb = dict(transpose=1, rounding=1, rht=1, sf_layout=nv.NVFP4_SF_ROWMAJOR)
    qa, qb = nv.nvfp4_quantize_dual(x.to(DEV), cfgs(**ma)[0], cfgs(**mb)[0])
    assert_quant_equal(qa, _oracle(x, ma))
    assert_quant_equal(qb, _oracle(x, mb))


def test_dual_unaligned_code_rows():
    # qk = 80 / 48: code rows of 40 / 24 bytes (not 16-byte multiples)
    x = syn.normal_bf16((48, 80), seed=45)
    ma, mb = dict(), dict(transpose=1, rounding=1)
    qa, qb = nv.nvfp4_quantize_dual(x.to(DEV), cfgs(**ma)[0], cfgs(**mb)[0])
    assert_quant_equal(qa, _oracle(x, ma))
    assert_quant_equal(qb, _oracle(x, mb))


def test_dual_rejects_bad_args():
    x = torch.zeros((32, 64), dtype=torch.bfloat16, device=DEV)
    ga = cfgs()[0]
    bad = cfgs(block=1, transpose=1)[0]
    bad.block = 7
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_quantize_dual(x, ga, bad)
    assert e.value.status == nv.NVFP4_ERR_INVALID_ARG
    # 16x16 blocks on Q = x^T need cols % 16 == 0 (qr = cols = 40 here)
    y = torch.zeros((32, 40), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_quantize_dual(y, ga, cfgs(block=1, transpose=1)[0])
    assert e.value.status == nv.NVFP4_ERR_UNSUPPORTED_SHAPE


def _extreme(kind, shape, seed):
    g = torch.Generator().manual_seed(seed)
    base = torch.randn(shape, generator=g)
    if kind == "tiny":        # amax ~1e-33: divisors below 2^-70 (IEEE-division path)
        x = base * 1e-34
    elif kind == "huge":      # amax ~1e37: divisors beyond 2^14 (IEEE division for stochastic rounding)
        x = base * 1e36
    elif kind == "mixed":     # 1e30-sized outliers next to 1e-30-sized elements in the same blocks
        x = base * 1e-30
        x[:, ::16] = base[:, ::16] * 1e30
    else:                     # subnormal BF16 elements next to ordinary ones
        x = base
        x[::2, 1::2] = base[::2, 1::2] * 1e-39
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("kind", ["tiny", "huge", "mixed", "subnormal"])
@pytest.mark.parametrize("mode", [dict(), dict(rounding=1), dict(rounding=1, rht=1), dict(block=1)],
                         ids=["rne", "sr", "sr-rht", "16x16"])
def test_extreme_ranges(kind, mode):
    x = _extreme(kind, (64, 192), seed=len(kind) * 101 + 7)
    assert torch.isfinite(x.float()).all()
    mb = dict(mode, transpose=1)
    qa, qb = nv.nvfp4_quantize_dual(x.to(DEV), cfgs(**mode)[0], cfgs(**mb)[0])
    assert_quant_equal(qa, _oracle(x, mode))
    assert_quant_equal(qb, _oracle(x, mb))


def test_dual_full_size_sampled():
    # dY of the MLP up-projection, both orientations as the training step
    # uses them; whole 16-row groups of each output checked against the oracle.
    _, _, dy = syn.config2()
    ma, mb = PAIRS["act-row-rne+col-sr-rht"]
    qa, qb = nv.nvfp4_quantize_dual(dy.to(DEV), cfgs(**ma)[0], cfgs(**mb)[0])
    u = syn.as_u16(dy)
    rng = np.random.default_rng(11)
    for q, m in ((qa, ma), (qb, mb)):
        n16 = q.rows // 16
        for gidx in (0, int(rng.integers(1, n16 - 1)), n16 - 1):
            r0 = gidx * 16
            ref = oracle.quantize_rows(u, cfgs(**m)[1], r0, r0 + 16)
            assert_quant_equal(q, ref, rows=np.arange(r0, r0 + 16))
