"""GPU Newton-Schulz step with NVFP4 products (Q-Root) against the oracle.

  * percentile of |x|, clipping and the FP32 combination: bit-exact on ragged
    sizes, with ties at the percentile, zeros, signed values and subnormals;
  * a three-step chain checked stage by stage: the oracle runs the chain, and
    each GPU stage is fed the oracle's own input of that stage (so every
    comparison is of the same computation): thresholds, clipped tensors,
    quantised operands and combinations bit-exact, every NVFP4 product within
    one BF16 ulp (at the GEMM tests' floor of 1e-3 of the largest output) of
    the oracle's FP64 GEMM of the same quantised operands;
  * nvfp4_ns_step itself equals the GPU composition of those stages bit for
    bit, stays within 1 % of the oracle's chain over three steps and within
    8 % of the same iteration in FP64 (the NVFP4 iteration error; the pages
    report about 3 % with clipping);
  * a signed partial permutation is a fixed point (a + b + c = 1, p = 100),
    exactly, as every NVFP4 step on it is exact.
"""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle

from _helpers import DEV, bf16_within_one_ulp

pytestmark = pytest.mark.gpu

QUINTIC = (15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0)


def _t(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(DEV)


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _f64(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


@pytest.mark.parametrize("n", [1, 7, 100, 1000, 12345, 65539, 1 << 20])
@pytest.mark.parametrize("p", [0.001, 50.0, 99.0, 99.9, 100.0])
def test_percentile_and_clip_bit_exact(n, p):
    rng = np.random.default_rng(n)
    v = rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))
    # ties: a tenth of the values share one magnitude, some zeros and subnormals
    v[rng.choice(n, size=max(1, n // 10), replace=False)] = -3.25
    v[rng.choice(n, size=max(1, n // 50), replace=False)] = 0.0
    v[rng.choice(n, size=max(1, n // 50), replace=False)] = 1e-39
    x = _bits(v)
    q_ref = oracle.abs_percentile_bf16(x, p)
    xd = _t(x)
    q = nv.nvfp4_abs_percentile_bf16(xd, p)
    assert q.cpu().numpy()[0].view(np.uint32) == np.float32(q_ref).view(np.uint32), (q.item(), q_ref)
    c = nv.nvfp4_clip_bf16(xd, q)
    assert np.array_equal(_u16(c), oracle.clip_bf16(x, q_ref))


def test_percentile_all_equal_and_sign_only():
    for vals in (np.full(4096, -2.0), np.full(4096, 0.0), np.tile([1.0, -1.0], 2048)):
        x = _bits(vals)
        for p in (1.0, 99.0, 100.0):
            q = nv.nvfp4_abs_percentile_bf16(_t(x), p).cpu().numpy()[0]
            assert np.float32(q) == oracle.abs_percentile_bf16(x, p)


@pytest.mark.parametrize("n", [8, 9, 4096, 100003])
def test_axpby_bit_exact(n):
    rng = np.random.default_rng(n)
    x = _bits(rng.standard_normal(n))
    y = _bits(rng.standard_normal(n) * 50)
    for a, b in ((1.875, -0.3125), (1.0, 1.0), (-2.5e-3, 7.0)):
        got = nv.nvfp4_axpby_bf16(_t(x), _t(y), a, b)
        assert np.array_equal(_u16(got), oracle.axpby_bf16(x, y, a, b))


def _quant_rows(xu16, transpose=False):
    cfg = nv.quant_cfg(transpose=1 if transpose else 0)
    return nv.nvfp4_quantize(_t(xu16), cfg)


def _assert_codes(q, xu16, transpose=False):
    from _helpers import assert_quant_equal
    assert_quant_equal(q, oracle.quantize(xu16, oracle.make_cfg(transpose=1 if transpose else 0)))


def _product_ok(lq, rq, l_u16, r_u16, r_transposed, ref_u16):
    """GPU BF16 product of the quantised operands against the oracle's FP64
    GEMM of its own quantisation of the same BF16 operands; the oracle's
    BF16 trace value must be that product rounded."""
    got = nv.nvfp4_gemm(lq, rq, out_dtype=nv.NVFP4_OUT_BF16).float().cpu().numpy()
    ol = oracle.quantize(l_u16, oracle.make_cfg())
    orr = oracle.quantize(r_u16, oracle.make_cfg(transpose=1 if r_transposed else 0))
    K = l_u16.shape[1]
    N = r_u16.shape[1] if r_transposed else r_u16.shape[0]
    ref = oracle.gemm_f64(ol, orr, l_u16.shape[0], N, K)
    assert np.array_equal(np.vectorize(oracle.bf16_rne_f64, otypes=[np.uint16])(ref), ref_u16)
    return bf16_within_one_ulp(got, ref)


@pytest.mark.parametrize("m,n", [(64, 192), (96, 160), (256, 1024)])
def test_chain_stage_by_stage(m, n):
    rng = np.random.default_rng(m * n)
    g = rng.standard_normal((m, n))
    x = _bits(g / np.linalg.norm(g))
    a, b, c = QUINTIC
    for step in range(3):
        out, tr = oracle.ns_step(x, a, b, c, p=99.0)
        # X: threshold, clip, both quantisations, A
        qx = nv.nvfp4_abs_percentile_bf16(_t(x), 99.0)
        assert np.float32(qx.item()) == tr["qx"]
        assert np.array_equal(_u16(nv.nvfp4_clip_bf16(_t(x), qx)), tr["xc"])
        q_rows, q_cols = _quant_rows(tr["xc"]), _quant_rows(tr["xc"], transpose=True)
        _assert_codes(q_rows, tr["xc"])
        _assert_codes(q_cols, tr["xc"], transpose=True)
        assert _product_ok(q_rows, q_rows, tr["xc"], tr["xc"], False, tr["a"]), ("A", step)
        # A A^T from the oracle's A
        qa = nv.nvfp4_abs_percentile_bf16(_t(tr["a"]), 99.0)
        assert np.float32(qa.item()) == tr["qa"]
        assert np.array_equal(_u16(nv.nvfp4_clip_bf16(_t(tr["a"]), qa)), tr["ac"])
        q_a = _quant_rows(tr["ac"])
        _assert_codes(q_a, tr["ac"])
        assert _product_ok(q_a, q_a, tr["ac"], tr["ac"], False, tr["a2"]), ("A2", step)
        # B and B X from the oracle's A, A2 and B
        assert np.array_equal(_u16(nv.nvfp4_axpby_bf16(_t(tr["a"]), _t(tr["a2"]), b, c)), tr["b"])
        qb = nv.nvfp4_abs_percentile_bf16(_t(tr["b"]), 99.0)
        assert np.float32(qb.item()) == tr["qb"]
        assert np.array_equal(_u16(nv.nvfp4_clip_bf16(_t(tr["b"]), qb)), tr["bc"])
        q_b = _quant_rows(tr["bc"])
        _assert_codes(q_b, tr["bc"])
        assert _product_ok(q_b, q_cols, tr["bc"], tr["xc"], True, tr["bx"]), ("BX", step)
        # X' from the oracle's X and B X
        assert np.array_equal(_u16(nv.nvfp4_axpby_bf16(_t(x), _t(tr["bx"]), a, 1.0)), out)
        x = out


def _composed_step(x, a, b, c, p):
    """nvfp4_ns_step spelled out with the library's own calls."""
    xc = nv.nvfp4_clip_bf16(x, nv.nvfp4_abs_percentile_bf16(x, p))
    q_rows, q_cols = nv.nvfp4_quantize_dual(xc, nv.quant_cfg(), nv.quant_cfg(transpose=1))
    A = nv.nvfp4_gemm(q_rows, q_rows, out_dtype=nv.NVFP4_OUT_BF16)
    q_a = nv.nvfp4_quantize(nv.nvfp4_clip_bf16(A, nv.nvfp4_abs_percentile_bf16(A, p)), nv.quant_cfg())
    A2 = nv.nvfp4_gemm(q_a, q_a, out_dtype=nv.NVFP4_OUT_BF16)
    B = nv.nvfp4_axpby_bf16(A, A2, b, c)
    q_b = nv.nvfp4_quantize(nv.nvfp4_clip_bf16(B, nv.nvfp4_abs_percentile_bf16(B, p)), nv.quant_cfg())
    BX = nv.nvfp4_gemm(q_b, q_cols, out_dtype=nv.NVFP4_OUT_BF16)
    return nv.nvfp4_axpby_bf16(x, BX, a, 1.0)


def _ns_fp64(x, a, b, c, steps):
    for _ in range(steps):
        A = x @ x.T
        x = a * x + (b * A + c * A @ A) @ x
    return x


@pytest.mark.parametrize("m,n", [(64, 192), (128, 512), (512, 2048)])
def test_ns_step_entry_point(m, n):
    rng = np.random.default_rng(m + n)
    g = rng.standard_normal((m, n))
    x0 = _bits(g / np.linalg.norm(g))
    x = _t(x0)
    ws = torch.zeros(nv.nvfp4_ns_workspace_size(m, n), dtype=torch.uint8, device=DEV)
    assert torch.equal(nv.nvfp4_ns_step(x, *QUINTIC, workspace=ws), _composed_step(x, *QUINTIC, 99.0))
    xo = x0
    for _ in range(3):
        x = nv.nvfp4_ns_step(x, *QUINTIC, workspace=ws)
        if m <= 128:
            xo, _ = oracle.ns_step(xo, *QUINTIC, p=99.0)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
    got = _f64(_u16(x))
    if m <= 128:
        ref = _f64(xo)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
    exact = _ns_fp64(_f64(x0), *QUINTIC, steps=3)
    assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < 0.08


def test_partial_permutation_fixed_point():
    m, n = 64, 256
    rng = np.random.default_rng(9)
    p = np.zeros((m, n), dtype=np.float32)
    p[np.arange(m), rng.permutation(n)[:m]] = rng.choice([-1.0, 1.0], size=m)
    x = _t(_bits(p))
    out = nv.nvfp4_ns_step(x, *QUINTIC, p=100.0)
    assert torch.equal(out, x)
    out2 = nv.nvfp4_ns_step(x, *(2 * v for v in QUINTIC), p=100.0)
    assert torch.equal(out2.float(), 2 * x.float())


def test_in_place_step():
    rng = np.random.default_rng(3)
    x = _t(_bits(rng.standard_normal((96, 224)) * 0.01))
    ref = nv.nvfp4_ns_step(x, *QUINTIC)
    y = x.clone()
    nv.nvfp4_ns_step(y, *QUINTIC, out=y)
    assert torch.equal(y, ref)
