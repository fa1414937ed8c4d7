"""The scratch-free quantiser entry point.

Some callers cannot allocate device memory (a host framework that owns every
allocation, code running inside another allocator's callbacks, paths that must
never reach an allocator), so nvfp4_quantize_noalloc keeps its scratch in a
file-scope device array instead of a caller workspace.  This test calls it
through the C ABI and checks it against nvfp4_quantize, bit for bit, on two
calls in a row with different inputs and configurations (the array keeps the
previous call's contents, which must not leak into the next result).  Errors
found on the device reach such callers only through the tensor scale (NaN):
non-finite input and a bounded wait that ran out are both checked here, each
followed by a clean call whose result must not be affected.  The file is named
to be collected last.
"""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _empty_like(q):
    return nv.NVFP4Tensor(codes=torch.empty_like(q.codes), sf=torch.empty_like(q.sf),
                          tensor_scale=torch.empty_like(q.tensor_scale), rows=q.rows, k=q.k, sf_layout=q.sf_layout)


def _same(a, b):
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.sf, b.sf)
    assert torch.equal(a.tensor_scale.view(torch.int32), b.tensor_scale.view(torch.int32))


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [
        (syn.normal_with_outliers_bf16((512, 1024), frac=0.01, seed=31),
         nv.quant_cfg(block=nv.NVFP4_BLOCK_16x16, rounding=nv.NVFP4_ROUND_RNE)),
        (syn.normal_bf16((384, 2048), std=3.0, seed=32),
         nv.quant_cfg(block=nv.NVFP4_BLOCK_1x16, rounding=nv.NVFP4_ROUND_SR, rht=1, transpose=1,
                      rht_seed=5, sr_seed=6, sr_offset=7)),
    ]
    for x_cpu, cfg in cases:
        x = x_cpu.cuda()
        ref = nv.nvfp4_quantize(x, cfg)
        out = _empty_like(ref)
        out.codes.fill_(0xAA)
        out.sf.fill_(0x55)
        nv.nvfp4_quantize_noalloc(x, cfg, out)
        torch.cuda.synchronize()
        _same(out, ref)


def test_noalloc_rejects_oversize_and_bad_args():
    import ctypes

    lib = nv.lib()
    P = ctypes.c_void_p
    cfg = nv.quant_cfg()
    big = lib.nvfp4_quantize_noalloc(P(8192), 1 << 17, 1 << 15, 1 << 15, ctypes.byref(cfg), P(8192), P(8192),
                                     P(8192), P(0))
    assert big == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_quantize_noalloc(P(8192), 64, 64, 64, None, P(8192), P(8192), P(8192), P(0)) == \
        nv.NVFP4_ERR_INVALID_ARG


def _check_clean_call(x, cfg):
    ref = nv.nvfp4_quantize(x, cfg)
    out = _empty_like(ref)
    nv.nvfp4_quantize_noalloc(x, cfg, out)
    torch.cuda.synchronize()
    _same(out, ref)


def test_noalloc_nonfinite_input_gives_nan_scale_then_clean_call():
    cfg = nv.quant_cfg(block=nv.NVFP4_BLOCK_1x16, rounding=nv.NVFP4_ROUND_RNE)
    x = syn.normal_bf16((256, 512), seed=33)
    bad = x.clone()
    bad[100, 37] = float("inf")
    bad[7, 500] = float("nan")
    xb = bad.cuda()
    ref = nv.nvfp4_quantize(x.cuda(), cfg)
    out = _empty_like(ref)
    nv.nvfp4_quantize_noalloc(xb, cfg, out)
    torch.cuda.synchronize()
    assert torch.isnan(out.tensor_scale).all()
    # the array's status word from the failed call must not leak
    _check_clean_call(x.cuda(), cfg)


@pytest.mark.parametrize("pass_", [1, 2], ids=["amax-pass", "encode-pass"])
def test_noalloc_timeout_gives_nan_scale_then_clean_call(pass_):
    cfg = nv.quant_cfg(block=nv.NVFP4_BLOCK_16x16, rounding=nv.NVFP4_ROUND_SR, rht=1, rht_seed=3, sr_seed=4)
    x = syn.normal_bf16((512, 768), seed=34).cuda()
    ref = nv.nvfp4_quantize(x, cfg)
    out = _empty_like(ref)
    nv.nvfp4_debug_quantize_skip_load(pass_)
    nv.nvfp4_quantize_noalloc(x, cfg, out)
    torch.cuda.synchronize()
    assert torch.isnan(out.tensor_scale).all()
    _check_clean_call(x, cfg)
