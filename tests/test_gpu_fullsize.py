"""Full-size parity of the benchmark step (the 12B MLP up-projection) and of
the 16384^3 roofline probe.

  * The three dual quantises the step runs -- X [8192, 5120] (rows RNE +
    columns RHT/SR), W [20480, 5120] (16x16 both ways) and dY [8192, 20480]
    (rows RNE + columns RHT/SR) -- are compared with the oracle's
    quantisation of the whole tensors, every code and scale byte.
  * Whole 256 x 256 output tiles of the fprop, dgrad and wgrad GEMMs and of
    16384^3 -- the first and last tiles, the middle one, and tiles on both
    sides of the persistent kernel's raster-group boundaries (groups of
    256-row or 256-column units sized to keep 32 MB of operand panels, the
    choice `_raster` repeats from the library's launcher) -- against the oracle's definition of the
    GEMM (FP64 sum of the products of its dequantised operands, the sum taken
    by a library FP64 matmul): BF16 output within one BF16 ulp at the floor
    of 1e-3 of the tile's largest value.
"""
import numpy as np
import pytest
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

from _helpers import DEV, assert_quant_equal, bf16_within_one_ulp

pytestmark = pytest.mark.gpu

T, HID, FFN = 8192, 5120, 20480
S = nv.NVFP4_DEFAULT_RHT_SEED
# the benchmark step's quantisations: (source, transpose, block, rounding, rht, sr_seed)
ROLES = {
    "x": ("x", 0, 0, 0, 0, 0), "xt": ("x", 1, 0, 1, 1, 6),
    "w": ("w", 0, 1, 0, 0, 0), "wt": ("w", 1, 1, 0, 0, 0),
    "dy": ("dy", 0, 0, 0, 0, 0), "dyt": ("dy", 1, 0, 1, 1, 5),
}
DUALS = [("x", "xt"), ("w", "wt"), ("dy", "dyt")]


def _cfgs(role):
    _, tr, block, rnd, rht, sr_seed = ROLES[role]
    g = nv.quant_cfg(block=block, rounding=rnd, rht=rht, transpose=tr, rht_seed=S, sr_seed=sr_seed)
    o = oracle.make_cfg(block=block, rounding=rnd, rht=rht, transpose=tr, rht_seed=S, sr_seed=sr_seed)
    return g, o


@pytest.fixture(scope="module")
def step():
    x, w, dy = syn.config2()
    src = {"x": x, "w": w, "dy": dy}
    gpu, ora = {}, {}
    for a, b in DUALS:
        ga, oa = _cfgs(a)
        gb, ob = _cfgs(b)
        xd = src[ROLES[a][0]].to(DEV)
        gpu[a], gpu[b] = nv.nvfp4_quantize_dual(xd, ga, gb)
        xu = syn.as_u16(src[ROLES[a][0]])
        ora[a] = oracle.quantize(xu, oa)
        ora[b] = oracle.quantize(xu, ob)
    torch.cuda.synchronize()
    return gpu, ora


@pytest.mark.parametrize("role", list(ROLES))
def test_step_quantisation_whole_tensor(step, role):
    gpu, ora = step
    assert_quant_equal(gpu[role], ora[role])


def _raster(M, N, K, budget=32.0e6):
    """The launcher's raster choice for a pair-mode GEMM: (groups of column
    blocks?, 256-row or 256-column units per group)."""
    a, b = M * K * 0.5625, N * K * 0.5625
    mu, tn = (M // 128 + 1) // 2, (N + 255) // 256
    gm = int(max(1.0, min(mu, budget * mu / a)))
    gn = int(max(1.0, min(tn, budget * tn / b)))
    by_m = a + b * ((mu + gm - 1) // gm)
    by_n = b + a * ((tn + gn - 1) // gn)
    return (True, gn) if by_n < by_m else (False, gm)


def _tiles(M, N, K, limit=12):
    """Top-left corners of 256 x 256 tiles to check: first, last, middle,
    then tiles on both sides of raster-group boundaries."""
    out = [(0, 0), (M - 256, N - 256), ((M // 2) // 256 * 256, (N // 2) // 256 * 256)]
    by_cols, g = _raster(M, N, K)
    for edge in range(g * 256, N if by_cols else M, g * 256):
        if by_cols:
            out += [(min(M - 256, 512), edge - 256), (min(M - 256, 256), edge)]
        else:
            out += [(edge - 256, min(N - 256, 768)), (edge, min(N - 256, 1024))]
    # the tiles on both sides of the end of the first persistent wave (76 CTA
    # pairs on 152 SMs), the first tile of the last wave and the last tile,
    # in the kernel's tile order: groups of g units along the grouped axis,
    # the grouped axis fastest inside a group (the last wave's tiles are the
    # ones a tail split cuts along K)
    mu, tn = M // 256, N // 256
    slow_n, fast_n = (mu, tn) if by_cols else (tn, mu)
    units = mu * tn
    waves = []
    for t in (75, 76, (units - 1) // 76 * 76, units - 1):
        if t >= units:
            continue
        grp, local = divmod(t, g * slow_n)
        first = grp * g
        gg = min(fast_n - first, g)
        fast, slow = first + local % gg, local // gg
        m, n = (slow, fast) if by_cols else (fast, slow)
        waves.append((m * 256, n * 256))
    out = out[:3] + waves + out[3:]
    seen = []
    for t in out:
        if t not in seen:
            seen.append(t)
    return seen[:limit]


def _check_tiles(d, qa, qb, M, N, K, tiles):
    dh = d.float().cpu().numpy()
    for r0, c0 in tiles:
        ac, asf, ascale = qa
        bc, bsf, bscale = qb
        da = oracle.dequantize(ac[r0:r0 + 256], asf[r0:r0 + 256], ascale, 256, K)
        db = oracle.dequantize(bc[c0:c0 + 256], bsf[c0:c0 + 256], bscale, 256, K)
        ref = da @ db.T
        assert bf16_within_one_ulp(dh[r0:r0 + 256, c0:c0 + 256], ref), (r0, c0)


@pytest.mark.parametrize("gemm", ["fprop", "dgrad", "wgrad"])
def test_step_gemm_whole_tiles(step, gemm):
    gpu, ora = step
    a, b, M, N, K = {"fprop": ("x", "w", T, FFN, HID), "dgrad": ("dy", "wt", T, HID, FFN),
                     "wgrad": ("dyt", "xt", FFN, HID, T)}[gemm]
    d = nv.nvfp4_gemm(gpu[a], gpu[b], out_dtype=nv.NVFP4_OUT_BF16)
    _check_tiles(d, ora[a], ora[b], M, N, K, _tiles(M, N, K))


def test_square_16k_whole_tiles():
    M = N = K = 16384
    a, b = syn.config4(M, N, K)
    g = nv.quant_cfg()
    qa = nv.nvfp4_quantize(a.to(DEV), g)
    qb = nv.nvfp4_quantize(b.to(DEV), g)
    d = nv.nvfp4_gemm(qa, qb, out_dtype=nv.NVFP4_OUT_BF16)
    tiles = _tiles(M, N, K, limit=8)
    rows_a = sorted({r for r, _ in tiles})
    rows_b = sorted({c for _, c in tiles})
    oc = oracle.make_cfg()
    au, bu = syn.as_u16(a), syn.as_u16(b)
    # quantise only the 256-row panels the tiles need (each call still takes
    # the whole operand's tensor scale)
    pa = {r: oracle.quantize_rows(au, oc, r, r + 256) for r in rows_a}
    pb = {c: oracle.quantize_rows(bu, oc, c, c + 256) for c in rows_b}
    dh = d.float().cpu().numpy()
    for r0, c0 in tiles:
        ac, asf, ascale = pa[r0]
        bc, bsf, bscale = pb[c0]
        ref = oracle.dequantize(ac, asf, ascale, 256, K) @ oracle.dequantize(bc, bsf, bscale, 256, K).T
        assert bf16_within_one_ulp(dh[r0:r0 + 256, c0:c0 + 256], ref), (r0, c0)
