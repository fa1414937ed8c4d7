"""The linear-layer wrappers (fprop, dgrad, wgrad) against the oracle: the
oracle quantises the same operands in the same orientation with the same
configuration, and its FP64 GEMM of those operands is the reference."""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import DEV, bf16_within_one_ulp, cfgs, rel_err

pytestmark = pytest.mark.gpu

RHT_SEED = 0x77AA


def _role_cfgs():
    # explicit configurations per operand role (transpose is set by the wrapper)
    x_f, _ = cfgs(block=0, rounding=0)
    w_f, _ = cfgs(block=1, rounding=0)
    dy_d, _ = cfgs(block=0, rounding=0)
    w_d, _ = cfgs(block=1, rounding=0)
    dy_w, _ = cfgs(block=0, rounding=1, rht=1, rht_seed=RHT_SEED, sr_seed=101)
    x_w, _ = cfgs(block=0, rounding=1, rht=1, rht_seed=RHT_SEED, sr_seed=202)
    return dict(fprop=(x_f, w_f), dgrad=(dy_d, w_d), wgrad=(dy_w, x_w))


def _ocfg(c, transpose):
    return oracle.make_cfg(block=c.block, rounding=c.rounding, rht=c.rht, transpose=transpose,
                           rht_seed=c.rht_seed, sr_seed=c.sr_seed, sr_offset=c.sr_offset)


def _run(op, x, w, dy, out_dtype):
    ca, cb = _role_cfgs()[op]
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    if op == "fprop":
        return nv.nvfp4_linear_fprop(xd, wd, ca, cb, out_dtype=out_dtype)
    if op == "dgrad":
        return nv.nvfp4_linear_dgrad(dyd, wd, ca, cb, out_dtype=out_dtype)
    return nv.nvfp4_linear_wgrad(dyd, xd, ca, cb, out_dtype=out_dtype)


def _operands(op, x, w, dy):
    """(A source, A transposed?, B source, B transposed?) as the wrapper
    quantises them."""
    if op == "fprop":
        return syn.as_u16(x), 0, syn.as_u16(w), 0
    if op == "dgrad":
        return syn.as_u16(dy), 0, syn.as_u16(w), 1
    return syn.as_u16(dy), 1, syn.as_u16(x), 1


def _reference_full(op, x, w, dy):
    ca, cb = _role_cfgs()[op]
    a_src, at, b_src, bt = _operands(op, x, w, dy)
    oa = oracle.quantize(a_src, _ocfg(ca, at))
    ob = oracle.quantize(b_src, _ocfg(cb, bt))
    M, N, K = oa[0].shape[0], ob[0].shape[0], oa[0].shape[1] * 2
    return oracle.gemm_f64(oa, ob, M, N, K)


@pytest.mark.parametrize("op", ["fprop", "dgrad", "wgrad"])
@pytest.mark.parametrize("T,din,dout", [(256, 256, 256), (96, 128, 384), (512, 160, 224)])
def test_small_full_compare(op, T, din, dout):
    x = syn.normal_bf16((T, din), seed=T + din)
    w = syn.normal_bf16((dout, din), std=0.02, seed=din + dout)
    dy = syn.normal_bf16((T, dout), std=1e-3, seed=T + dout)
    ref = _reference_full(op, x, w, dy)
    got = _run(op, x, w, dy, nv.NVFP4_OUT_F32).cpu().numpy()
    assert rel_err(got, ref) <= 1e-3
    got_bf = _run(op, x, w, dy, nv.NVFP4_OUT_BF16).float().cpu().numpy()
    assert bf16_within_one_ulp(got_bf, ref)


def test_default_configurations_are_the_documented_ones():
    T, din, dout = 128, 128, 256
    x = syn.normal_bf16((T, din), seed=1).to(DEV)
    w = syn.normal_bf16((dout, din), std=0.02, seed=2).to(DEV)
    dy = syn.normal_bf16((T, dout), std=1e-3, seed=3).to(DEV)
    s = nv.NVFP4_DEFAULT_RHT_SEED
    pairs = [
        (nv.nvfp4_linear_fprop, (x, w), nv.quant_cfg(block=0), nv.quant_cfg(block=1)),
        (nv.nvfp4_linear_dgrad, (dy, w), nv.quant_cfg(block=0), nv.quant_cfg(block=1)),
        (nv.nvfp4_linear_wgrad, (dy, x), nv.quant_cfg(rounding=1, rht=1, rht_seed=s, sr_seed=5),
         nv.quant_cfg(rounding=1, rht=1, rht_seed=s, sr_seed=6)),
    ]
    for fn, args, ca, cb in pairs:
        a = fn(*args, out_dtype=nv.NVFP4_OUT_F32)
        b = fn(*args, ca, cb, out_dtype=nv.NVFP4_OUT_F32)
        assert torch.equal(a, b), fn.__name__


def test_weight_transpose_property_on_gpu():
    # dgrad quantises W^T with 16x16 tiles; that must equal the nibble-wise
    # transpose of W's own 16x16 quantisation.
    w = syn.normal_with_outliers_bf16((256, 384), frac=0.01, seed=9).to(DEV)
    g0, _ = cfgs(block=1, sf_layout=nv.NVFP4_SF_ROWMAJOR)
    g1, _ = cfgs(block=1, transpose=1, sf_layout=nv.NVFP4_SF_ROWMAJOR)
    q0 = nv.nvfp4_quantize(w, g0)
    q1 = nv.nvfp4_quantize(w, g1)
    c0 = q0.codes.cpu().numpy()
    c1 = q1.codes.cpu().numpy()
    u0 = np.empty((256, 384), np.uint8)
    u0[:, 0::2], u0[:, 1::2] = c0 & 15, c0 >> 4
    u1 = np.empty((384, 256), np.uint8)
    u1[:, 0::2], u1[:, 1::2] = c1 & 15, c1 >> 4
    assert np.array_equal(u0.T, u1)
    s0 = q0.sf.cpu().numpy()[: 256 * 24].reshape(256, 24)
    s1 = q1.sf.cpu().numpy()[: 384 * 16].reshape(384, 16)
    assert np.array_equal(s0[::16, :].T, s1[::16, :])
    assert q0.tensor_scale.item() == q1.tensor_scale.item()


def _sampled(op, x, w, dy, d, out_f32, nblocks=3):
    ca, cb = _role_cfgs()[op]
    a_src, at, b_src, bt = _operands(op, x, w, dy)
    oca, ocb = _ocfg(ca, at), _ocfg(cb, bt)
    M, N = d.shape
    rng = np.random.default_rng(17)
    picks = [(0, 0), (M - 16, N - 16)] + [(int(rng.integers(0, M // 16)) * 16, int(rng.integers(0, N // 16)) * 16)
                                          for _ in range(nblocks - 2)]
    for r0, c0 in picks:
        oa = oracle.quantize_rows(a_src, oca, r0, r0 + 16)
        ob = oracle.quantize_rows(b_src, ocb, c0, c0 + 16)
        K = oa[0].shape[1] * 2
        ref = oracle.gemm_f64(oa, ob, 16, 16, K)
        got = d[r0:r0 + 16, c0:c0 + 16].float().cpu().numpy()
        if out_f32:
            assert rel_err(got, ref) <= 1e-3, (op, r0, c0)
        else:
            assert bf16_within_one_ulp(got, ref), (op, r0, c0)


@pytest.mark.parametrize("op", ["fprop", "dgrad", "wgrad"])
def test_mlp_up_12b_sampled(op):
    x, w, dy = syn.config2()
    d = _run(op, x, w, dy, nv.NVFP4_OUT_BF16)
    _sampled(op, x, w, dy, d, out_f32=False)


@pytest.mark.parametrize("name", ["qkv", "mlp_up", "mlp_down"])
def test_projections_3b_chain_sampled(name):
    x, w, dy = syn.config3(name)
    for op in ("fprop", "dgrad", "wgrad"):
        d = _run(op, x, w, dy, nv.NVFP4_OUT_F32)
        _sampled(op, x, w, dy, d, out_f32=True, nblocks=2)
