"""GPU GEMM parity with the oracle's FP64 accumulation of the same dequantised
operands: FP32 output within max relative error 1e-3 (floored at 1e-3 of the
largest output), BF16 output within one BF16 ulp; hand-built unit-scale
operands must match exactly (which pins nibble order and the scale layout
independently of any tolerance)."""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import DEV, bf16_within_one_ulp, cfgs, rel_err

pytestmark = pytest.mark.gpu

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _pack(c4):
    return (c4[:, 0::2] | (c4[:, 1::2] << 4)).astype(np.uint8)


def _grid_values(c4):
    mag = GRID[c4 & 7]
    return np.where(c4 & 8, -mag, mag)


def _operand(codes, sf_rowmajor, scale, rows, k):
    return nv.NVFP4Tensor(
        codes=torch.from_numpy(codes).to(DEV),
        sf=torch.from_numpy(oracle.sf_to_mma(sf_rowmajor, rows, k)).to(DEV),
        tensor_scale=torch.tensor([scale], dtype=torch.float32, device=DEV),
        rows=rows, k=k, sf_layout=nv.NVFP4_SF_MMA)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (128, 256, 256), (256, 256, 256), (200, 300, 96),
                                   (1, 1, 32), (128, 512, 1024), (300, 700, 2080), (512, 512, 8192),
                                   (384, 300, 10240)])
def test_unit_scales_exact(M, N, K):
    # (the last two are cut along K into pieces, one per CTA pair: integer
    # quarters keep every partial sum exact, so any summation order matches)
    rng = np.random.default_rng(M + N + K)
    ca = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
    cb = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    one_a = np.full((M, K // 16), 0x38, dtype=np.uint8)
    one_b = np.full((N, K // 16), 0x38, dtype=np.uint8)
    a = _operand(_pack(ca), one_a, 1.0, M, K)
    b = _operand(_pack(cb), one_b, 1.0, N, K)
    d = nv.nvfp4_gemm(a, b, out_dtype=nv.NVFP4_OUT_F32).cpu().numpy().astype(np.float64)
    ref = _grid_values(ca) @ _grid_values(cb).T
    if not np.array_equal(d, ref):
        bad = np.argwhere(d != ref)
        m, n = bad[0]
        raise AssertionError("%d mismatches; first (%d,%d): gpu %r exact %r" % (len(bad), m, n, d[m, n], ref[m, n]))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 300, 96), (384, 512, 1024)])
def test_single_scale_per_row_and_k_block(M, N, K):
    # Distinct scale per (row, 16-block) with unit codes isolates the scale
    # layout: D[m, n] = sum_kb 16 * sfA[m,kb] * sfB[n,kb] for all-ones codes.
    rng = np.random.default_rng(1)
    sfa = rng.integers(0x30, 0x48, size=(M, K // 16), dtype=np.uint8)
    sfb = rng.integers(0x30, 0x48, size=(N, K // 16), dtype=np.uint8)
    ones = np.full((M, K), 2, dtype=np.uint8)  # code 2 = 1.0
    onesb = np.full((N, K), 2, dtype=np.uint8)
    a = _operand(_pack(ones), sfa, 1.0, M, K)
    b = _operand(_pack(onesb), sfb, 1.0, N, K)
    d = nv.nvfp4_gemm(a, b, out_dtype=nv.NVFP4_OUT_F32).cpu().numpy().astype(np.float64)
    e4 = np.vectorize(oracle.e4m3_value)
    ref = 16.0 * (e4(sfa) @ e4(sfb).T)
    assert rel_err(d, ref) <= 1e-6


def _quantised(x, **mode):
    g, o = cfgs(**mode)
    q = nv.nvfp4_quantize(x.to(DEV), g)
    return q, oracle.quantize(syn.as_u16(x), o)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (130, 260, 320), (383, 513, 544), (64, 1000, 128),
                                   (383, 520, 544), (1000, 776, 256)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_quantised_operands_vs_oracle(M, N, K, out):
    a = syn.normal_bf16((M, K), seed=M)
    b = syn.normal_bf16((N, K), seed=N + 1)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b, block=0, rounding=1, rht=1)
    ref = oracle.gemm_f64(oa, ob, M, N, K)
    if out == "f32":
        d = nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_F32).cpu().numpy()
        assert rel_err(d, ref) <= 1e-3
    else:
        d = nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_BF16).float().cpu().numpy()
        assert bf16_within_one_ulp(d, ref)


def test_config0_fprop_fp32():
    x, w = syn.config0()
    qx, ox = _quantised(x)
    qw, ow = _quantised(w)
    d = nv.nvfp4_gemm(qx, qw, out_dtype=nv.NVFP4_OUT_F32).cpu().numpy()
    assert rel_err(d, oracle.gemm_f64(ox, ow, 256, 256, 256)) <= 1e-3


def test_padded_output_stride_bf16_clipped():
    # BF16 output through the staged (TMA) store path with a padded row
    # stride and a D view shorter than its buffer: ragged row and column
    # boxes must be clipped at M and N, nothing written outside.
    M, N, K = 200, 200, 256
    a = syn.normal_bf16((M, K), seed=5)
    b = syn.normal_bf16((N, K), seed=6)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b)
    big = torch.full((M + 40, 264), 7.0, dtype=torch.bfloat16, device=DEV)
    nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_BF16, d=big[:M, :N])
    host = big.float().cpu().numpy()
    assert np.all(host[:, N:] == 7.0) and np.all(host[M:, :] == 7.0)
    assert bf16_within_one_ulp(host[:M, :N], oracle.gemm_f64(oa, ob, M, N, K))


def test_padded_output_stride():
    a = syn.normal_bf16((128, 256), seed=3)
    b = syn.normal_bf16((256, 256), seed=4)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b)
    big = torch.full((128, 300), 7.0, dtype=torch.float32, device=DEV)
    nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_F32, d=big)
    host = big.cpu().numpy()
    assert np.all(host[:, 256:] == 7.0)  # nothing written past N
    assert rel_err(host[:, :256], oracle.gemm_f64(oa, ob, 128, 256, 256)) <= 1e-3


def _sampled_check(qa, qb, a_cpu, b_cpu, d, out_f32, a_mode=None, b_mode=None, blocks=((0, 0), (1, 1), (-1, -1))):
    """Compare 16x16 output blocks with the oracle, quantising only the rows
    those blocks need."""
    _, oa_cfg = cfgs(**(a_mode or {}))
    _, ob_cfg = cfgs(**(b_mode or {}))
    M, N, K = qa.rows, qb.rows, qa.k
    au, bu = syn.as_u16(a_cpu), syn.as_u16(b_cpu)
    rng = np.random.default_rng(5)
    for bm, bn in blocks:
        r0 = (M - 16) if bm < 0 else (int(rng.integers(0, M // 16)) * 16 if bm > 0 else 0)
        c0 = (N - 16) if bn < 0 else (int(rng.integers(0, N // 16)) * 16 if bn > 0 else 0)
        oa = oracle.quantize_rows(au, oa_cfg, r0, r0 + 16)
        ob = oracle.quantize_rows(bu, ob_cfg, c0, c0 + 16)
        ref = oracle.gemm_f64(oa, ob, 16, 16, K)
        got = d[r0:r0 + 16, c0:c0 + 16].float().cpu().numpy()
        if out_f32:
            assert rel_err(got, ref) <= 1e-3, (r0, c0)
        else:
            assert bf16_within_one_ulp(got, ref), (r0, c0)


def test_many_tiles_per_cta():
    M, N, K = 4096, 4096, 256  # 512 tiles: several per persistent CTA
    a = syn.normal_bf16((M, K), seed=11)
    b = syn.normal_bf16((N, K), seed=12)
    qa, _ = _quantised(a)
    qb, _ = _quantised(b)
    d = nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_F32)
    _sampled_check(qa, qb, a, b, d, True, blocks=((0, 0), (1, 1), (1, 1), (1, 1), (-1, -1)))


@pytest.mark.parametrize("M,N,K", [(16384, 16384, 16384), (128, 8192, 8192)], ids=["square16k", "skinny"])
def test_roofline_probe_shapes_sampled(M, N, K):
    a, b = syn.config4(M, N, K)
    qa, _ = _quantised(a)
    qb, _ = _quantised(b)
    d = nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_BF16)
    _sampled_check(qa, qb, a, b, d, False)


def test_timeout_is_reported_and_context_survives():
    a = syn.normal_bf16((512, 1024), seed=21)
    b = syn.normal_bf16((512, 1024), seed=22)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b)
    ws = torch.zeros(nv.nvfp4_gemm_workspace_size(512, 512, 1024), dtype=torch.uint8, device=DEV)
    nv.nvfp4_debug_gemm_skip_load(True)
    nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_F32, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_ERR_TIMEOUT
    # the hook is one-shot and the context is still usable
    d = nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_F32, workspace=ws)
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
    assert rel_err(d.cpu().numpy(), oracle.gemm_f64(oa, ob, 512, 512, 1024)) <= 1e-3


def test_dequantize_matches_oracle():
    x = syn.normal_with_outliers_bf16((96, 512), frac=0.01, seed=8)
    for layout in (nv.NVFP4_SF_MMA, nv.NVFP4_SF_ROWMAJOR):
        g, o = cfgs(sf_layout=layout, rounding=1, rht=1)
        q = nv.nvfp4_quantize(x.to(DEV), g)
        oc = oracle.quantize(syn.as_u16(x), o)
        ref = oracle.dequantize(*oc, 96, 512)
        f32 = nv.nvfp4_dequantize(q, nv.NVFP4_OUT_F32).cpu().numpy()
        assert np.array_equal(f32, ref.astype(np.float32))
        bf = nv.nvfp4_dequantize(q, nv.NVFP4_OUT_BF16).cpu()
        assert torch.equal(bf, torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16))


def test_empty_shapes():
    g, _ = cfgs()
    a = nv.nvfp4_quantize(torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV), g)
    b = nv.nvfp4_quantize(syn.normal_bf16((32, 64), seed=1).to(DEV), g)
    d = nv.nvfp4_gemm(a, b, out_dtype=nv.NVFP4_OUT_F32)
    torch.cuda.synchronize()
    assert d.shape == (0, 32)


@pytest.mark.parametrize("M,N,K", [(128, 8192, 8192), (100, 1000, 4160), (1, 256, 8192), (64, 520, 2048),
                                   (128, 2304, 16384)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_split_k_vs_oracle(M, N, K, out):
    # one row block with few tiles: the workspace from nvfp4_gemm_workspace_size
    # holds split-K scratch, and the header-only workspace runs unsplit
    a = syn.normal_bf16((M, K), seed=M + 7)
    b = syn.normal_bf16((N, K), seed=N + 8)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b, block=0, rounding=1, rht=1)
    od = nv.NVFP4_OUT_F32 if out == "f32" else nv.NVFP4_OUT_BF16
    ws = torch.zeros(nv.nvfp4_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    assert ws.numel() > 256, "this shape is expected to split"
    d = nv.nvfp4_gemm(qa, qb, out_dtype=od, workspace=ws)
    d_plain = nv.nvfp4_gemm(qa, qb, out_dtype=od, workspace=torch.zeros(256, dtype=torch.uint8, device=DEV))
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
    # the oracle's GEMM definition (FP64 sum over its dequantised operands),
    # summed by a library FP64 matmul for these long shapes
    ref = oracle.dequantize(*oa, M, K) @ oracle.dequantize(*ob, N, K).T
    for got in (d, d_plain):
        g = got.float().cpu().numpy()
        if out == "f32":
            assert rel_err(g, ref) <= 1e-3
        else:
            assert bf16_within_one_ulp(g, ref)


def test_mma_rate_measurement_runs():
    # the roofline measurement completes cleanly and gives plausible rates
    for kind in nv.MMA_RATE_KINDS:
        tf, cyc = nv.nvfp4_debug_mma_rate(kind, 256)
        assert 16.0 < cyc < 4096.0, (kind, cyc)
        assert 50.0 < tf < 50000.0, (kind, tf)


def _tail_plan(M, N, K, clusters):
    """The tail split nvfp4_gemm documents (include/nvfp4.h): tiles past the
    last whole wave of CTA pairs, when they would leave at least half the
    pairs idle, cut along K into whole groups of four 256-wide k-blocks, one
    piece per pair, if that takes at least 24 k-blocks off the last wave."""
    kb = -(-K // 256)
    units = -(-M // 256) * -(-N // 256)
    rem = units % clusters
    if rem == 0 or kb < 8:
        return 0, 0, 0
    s = min(clusters // rem, kb // 4)
    if s < 2:
        return 0, 0, 0
    per = -(-(-(-kb // s)) // 4) * 4
    s = -(-kb // per)
    if s < 2 or kb - per < 24:
        return 0, 0, 0
    return rem, s, per


def _pair_clusters():
    # CTA pairs the persistent GEMM launches on a shape with many tiles
    return nv.nvfp4_gemm_plan(16384, 16384, 1024)["ctas"] // 2


@pytest.mark.parametrize("shape", ["all-split", "last-wave", "odd-rows"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_tail_split_vs_oracle(shape, out):
    C = _pair_clusters()
    if shape == "all-split":      # fewer tiles than pairs: every tile cut along K
        M, N, K = 512, 512, 8192
    elif shape == "last-wave":    # one whole wave, then a few tiles cut; ragged rows, columns and K
        M, N, K = 256 * (C // 10 + 1) - 200, 2404, 8320
    else:                         # odd row blocks: the second pair's follower lies past M
        M, N, K = 384, 300, 10240
    tiles, split, per = _tail_plan(M, N, K, C)
    assert tiles > 0, "this shape is expected to split"
    plan = nv.nvfp4_gemm_plan(M, N, K)
    assert plan["pair"] == 1 and (plan["tail_tiles"], plan["tail_split"], plan["tail_kb"]) == (tiles, split, per)
    assert nv.nvfp4_gemm_plan(M, N, K, 256)["tail_tiles"] == 0  # header-only workspace: unsplit
    a = syn.normal_bf16((M, K), seed=M + 17)
    b = syn.normal_bf16((N, K), seed=N + 18)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b, block=0, rounding=1, rht=1)
    od = nv.NVFP4_OUT_F32 if out == "f32" else nv.NVFP4_OUT_BF16
    ws = torch.zeros(nv.nvfp4_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    d = nv.nvfp4_gemm(qa, qb, out_dtype=od, workspace=ws)
    d_plain = nv.nvfp4_gemm(qa, qb, out_dtype=od, workspace=torch.zeros(256, dtype=torch.uint8, device=DEV))
    assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
    # the oracle's GEMM definition (FP64 sum over its dequantised operands),
    # summed by a library FP64 matmul for these long shapes
    ref = oracle.dequantize(*oa, M, K) @ oracle.dequantize(*ob, N, K).T
    for got in (d, d_plain):
        g = got.float().cpu().numpy()
        if out == "f32":
            assert rel_err(g, ref) <= 1e-3
        else:
            assert bf16_within_one_ulp(g, ref)



@pytest.mark.parametrize("pitch", [528, 523], ids=["aligned-rows", "odd-rows"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_tail_split_padded_output(pitch, out):
    # the K-split tiles' reduction writes D through a padded row stride (16-byte
    # rows: vector stores; odd pitch: element stores) and nothing past M or N
    M, N, K = 512, 520, 8192
    assert nv.nvfp4_gemm_plan(M, N, K)["tail_tiles"] > 0, "this shape is expected to split"
    a = syn.normal_bf16((M, K), seed=31)
    b = syn.normal_bf16((N, K), seed=32)
    qa, oa = _quantised(a)
    qb, ob = _quantised(b)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    big = torch.full((M + 8, pitch), 7.0, dtype=dt, device=DEV)
    nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_F32 if out == "f32" else nv.NVFP4_OUT_BF16, d=big[:M, :N])
    host = big.float().cpu().numpy()
    assert np.all(host[:, N:] == 7.0) and np.all(host[M:, :] == 7.0)
    ref = oracle.dequantize(*oa, M, K) @ oracle.dequantize(*ob, N, K).T
    if out == "f32":
        assert rel_err(host[:M, :N], ref) <= 1e-3
    else:
        assert bf16_within_one_ulp(host[:M, :N], ref)
