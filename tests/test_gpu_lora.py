"""GPU LoRA-SVD projection forward against the oracle.

The forward is Y = Q(X) Q(W_res)^T + beta U L2^T with U = BF16(X L1^T)
("Full-Stack FP4...", section 2.1).  What is checked:
  * U: the GPU accumulates X L1^T in FP32 on the tensor cores, the oracle in
    FP64, so the two BF16 roundings may differ where the FP32 sum and the
    exact one round differently -- near a rounding midpoint, or anywhere in a
    sum that nearly cancels (its relative error is then large).  Every GPU
    element must equal the oracle's, or be within half a BF16 ulp of a value
    that lies within the summation bound din 2^-22 sum_k |x_k| |l1_k| of the
    exact sum (four times the textbook FP32 bound, for the tensor cores'
    accumulation order);
  * Y: within the GEMM tolerance (FP32 output: max relative error 1e-3 floored
    at 1e-3 of the largest output; BF16 output: one BF16 ulp at that floor),
    plus two terms the branch's arithmetic brings: the library adds it to the
    NVFP4 accumulator as hi + lo = (beta / (sX sW)) U in two BF16 parts, which
    carry it to 2^-18 relative (each part's rounding is 2^-9 of what it
    represents) plus three FP32 roundings (2^-24 each), so 2^-16 |beta|
    sum_j |U_j| |L2_nj| bounds it with margin; and, in rows where U
    legitimately differs, |beta| sum_j |dU_j| |L2_nj|;
  * beta = 0 gives exactly the plain NVFP4 GEMM;
  * the 12B MLP up-projection shape, sampled.
The oracle quantises X and W_res itself (its codes equal the GPU's bit for
bit, as the quantiser tests establish) and computes Y from its own operands.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import DEV, cfgs

pytestmark = pytest.mark.gpu


def _bf16_f64(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _inputs(T, din, dout, r, seed):
    x = syn.normal_bf16((T, din), seed=seed)
    w = syn.normal_bf16((dout, din), std=0.02, seed=seed + 1)
    l1 = syn.normal_bf16((r, din), std=0.05, seed=seed + 2)
    l2 = syn.normal_bf16((dout, r), std=0.05, seed=seed + 3)
    return x, w, l1, l2


def _w_block(dout):
    # the weight's 16x16 blocks need dout % 16 == 0; ragged test shapes use 1x16
    return 1 if dout % 16 == 0 else 0


def _gpu(x, w, l1, l2, beta, out_dtype):
    gx, _ = cfgs(block=0)
    gw, _ = cfgs(block=_w_block(w.shape[0]))
    xq = nv.nvfp4_quantize(x.to(DEV), gx)
    wq = nv.nvfp4_quantize(w.to(DEV), gw)
    y, u = nv.nvfp4_lora_forward(xq, wq, x.to(DEV), l1.to(DEV), l2.to(DEV), beta, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return xq, wq, y, u


def _check_u(u_gpu, u_ref, u_exact, x_f64, l1_f64):
    """u_*: uint16 [rows, r]; u_exact FP64 sums; x_f64 [rows, din], l1_f64
    [r, din].  Returns |U_gpu - U_ref| as FP64."""
    din = x_f64.shape[1]
    g = _bf16_f64(u_gpu)
    diff = np.argwhere(u_gpu != u_ref)
    assert len(diff) <= max(8, u_gpu.size // 20), "too many U mismatches: %d of %d" % (len(diff), u_gpu.size)
    if len(diff):
        absdot = np.abs(x_f64) @ np.abs(l1_f64).T
        bound = din * 2.0 ** -22 * absdot
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(g), 2.0 ** -133))) - 8)
        for t, j in diff:
            assert abs(g[t, j] - u_exact[t, j]) <= bound[t, j] + half_ulp[t, j], \
                (t, j, hex(int(u_gpu[t, j])), hex(int(u_ref[t, j])), u_exact[t, j], bound[t, j])
    return np.abs(g - _bf16_f64(u_ref))


def _branch_bound(beta, u_ref_u16, l2_u16):
    """2^-16 |beta| sum_j |U_j| |L2_nj|: the hi / lo representation of the
    branch inside the FP32 accumulator (see the module docstring)."""
    return 2.0 ** -16 * abs(beta) * (np.abs(_bf16_f64(u_ref_u16)) @ np.abs(_bf16_f64(l2_u16)).T)


def _check_y(got, ref, extra, bf16):
    got = np.asarray(got, np.float64)
    floor = 1e-3 * max(np.abs(ref).max(), 1e-300)
    mag = np.maximum(np.abs(ref), floor)
    if bf16:
        allow = np.exp2(np.floor(np.log2(mag)) - 7)
    else:
        allow = 1e-3 * mag
    err = np.abs(got - ref)
    bad = err > allow + 1.001 * extra
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError("Y: %d elements outside tolerance; first %s: got %r ref %r err %.3g allow %.3g "
                             "extra %.3g max|ref| %.3g" % (bad.sum(), i, got[i], ref[i], err[i], allow[i], extra[i],
                                                          np.abs(ref).max()))


CASES = [  # T, din, dout, r, beta, out
    (256, 256, 256, 64, 1.0, "f32"),
    (200, 320, 300, 40, -0.75, "f32"),
    (130, 128, 520, 128, 2.5, "bf16"),
    (96, 64, 64, 8, 0.3, "f32"),       # one row block: single-CTA GEMM mode
    (384, 512, 768, 256, 1.0, "bf16"),
    (1000, 160, 136, 72, 0.5, "f32"),
]


@pytest.mark.parametrize("T,din,dout,r,beta,out", CASES, ids=lambda v: str(v))
def test_lora_forward_vs_oracle(T, din, dout, r, beta, out):
    x, w, l1, l2 = _inputs(T, din, dout, r, seed=T + din + r)
    od = nv.NVFP4_OUT_F32 if out == "f32" else nv.NVFP4_OUT_BF16
    _, _, y, u = _gpu(x, w, l1, l2, beta, od)
    xu, wu, l1u, l2u = (syn.as_u16(t) for t in (x, w, l1, l2))
    _, ox = cfgs(block=0)
    _, ow = cfgs(block=_w_block(dout))
    xq_o = oracle.quantize(xu, ox)
    wq_o = oracle.quantize(wu, ow)
    u_ref, u_exact = oracle.lora_down(xu, l1u)
    du = _check_u(u.view(torch.int16).cpu().numpy().view(np.uint16), u_ref, u_exact, _bf16_f64(xu), _bf16_f64(l1u))
    ref = oracle.lora_forward(xq_o, wq_o, xu, l1u, l2u, beta)
    extra = abs(beta) * (du @ np.abs(_bf16_f64(l2u)).T) + _branch_bound(beta, u_ref, l2u)
    _check_y(y.float().cpu().numpy(), ref, extra, out == "bf16")
    # the branch is not negligible in these cases
    plain = oracle.gemm_f64(xq_o, wq_o, T, dout, din)
    assert np.abs(ref - plain).max() > 0.05 * np.abs(ref).max()


def test_beta_zero_is_the_plain_gemm():
    x, w, l1, l2 = _inputs(300, 256, 384, 64, seed=77)
    for od in (nv.NVFP4_OUT_F32, nv.NVFP4_OUT_BF16):
        xq, wq, y, _ = _gpu(x, w, l1, l2, 0.0, od)
        plain = nv.nvfp4_gemm(xq, wq, out_dtype=od)
        assert torch.equal(y, plain)


def test_mlp_up_shape_sampled():
    T, din, dout, r = 8192, 5120, 20480, 64
    x, w, _ = syn.config2(tokens=T, hidden=din, ffn=dout)
    l1 = syn.normal_bf16((r, din), std=0.02, seed=91)
    l2 = syn.normal_bf16((dout, r), std=0.02, seed=92)
    _, _, y, u = _gpu(x, w, l1, l2, 1.0, nv.NVFP4_OUT_BF16)
    xu, wu, l1u, l2u = (syn.as_u16(t) for t in (x, w, l1, l2))
    _, ox = cfgs(block=0)
    _, ow = cfgs(block=1)
    ug = u.view(torch.int16).cpu().numpy().view(np.uint16)
    yh = y.float().cpu().numpy()
    rng = np.random.default_rng(93)
    # 16 x 16 blocks in the first, a middle and the last tile rows / columns
    for r0, c0 in ((0, 0), (int(rng.integers(1, T // 16 - 1)) * 16, int(rng.integers(1, dout // 16 - 1)) * 16),
                   (T - 16, dout - 16), (4096, 10240 + 128)):
        xr = xu[r0:r0 + 16]
        u_ref, u_exact = oracle.lora_down(xr, l1u)
        du = _check_u(ug[r0:r0 + 16], u_ref, u_exact, _bf16_f64(xr), _bf16_f64(l1u))
        xq_o = oracle.quantize_rows(xu, ox, r0, r0 + 16)
        wq_o = oracle.quantize_rows(wu, ow, c0, c0 + 16)
        tt, nn = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
        ref = oracle.lora_forward_sampled(xq_o, wq_o, xr, l1u, l2u[c0:c0 + 16], 1.0, tt.ravel(),
                                          nn.ravel()).reshape(16, 16)
        extra = du @ np.abs(_bf16_f64(l2u[c0:c0 + 16])).T + _branch_bound(1.0, u_ref, l2u[c0:c0 + 16])
        _check_y(yh[r0:r0 + 16, c0:c0 + 16], ref, extra, True)


def test_lora_rejects_bad_shapes():
    lib = nv.lib()
    P = ctypes.c_void_p
    x, w, l1, l2 = _inputs(64, 64, 64, 16, seed=5)
    gx, _ = cfgs()
    xq = nv.nvfp4_quantize(x.to(DEV), gx)
    wq = nv.nvfp4_quantize(w.to(DEV), gx)
    ta, tb = xq._c(), wq._c()
    for r in (4, 12, 264):
        assert lib.nvfp4_lora_forward(ctypes.byref(ta), ctypes.byref(tb), P(8192), 64, P(8192), P(8192), r, 1.0, 0,
                                      P(8192), 64, P(8192), P(8192), 1 << 20, P(0)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
