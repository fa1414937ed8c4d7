"""Shared test helpers: run the CUDA path through the C ABI and compare with
the oracle.  (Test infrastructure; the oracle is imported only here and in
the tests.)"""
import numpy as np
import torch

import block_scaled_gemm_nvfp4_gb300 as nv
import oracle
from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

DEV = "cuda"

ALL_MODES = [dict(block=b, rounding=r, rht=h) for b in (0, 1) for r in (0, 1) for h in (0, 1)]


def mode_id(m):
    return "%s-%s-%s" % ("16x16" if m["block"] else "1x16", "sr" if m["rounding"] else "rne",
                         "rht" if m["rht"] else "plain")


def cfgs(block=0, rounding=0, rht=0, transpose=0, rht_seed=0x1234ABCD, sr_seed=0xC0FFEE, sr_offset=7,
         sf_layout=nv.NVFP4_SF_MMA):
    g = nv.quant_cfg(block=block, rounding=rounding, rht=rht, sf_layout=sf_layout, transpose=transpose,
                     rht_seed=rht_seed, sr_seed=sr_seed, sr_offset=sr_offset)
    o = oracle.make_cfg(block=block, rounding=rounding, rht=rht, transpose=transpose, rht_seed=rht_seed,
                        sr_seed=sr_seed, sr_offset=sr_offset)
    return g, o


def sf_rows_from_mma(sf_mma, rows, kb_count, qk):
    """Gather row-major scales for the given rows out of the tensor-core
    layout, using the oracle's statement of that layout."""
    idx = np.array([[oracle.sf_mma_offset(r, kb, qk) for kb in range(kb_count)] for r in rows], dtype=np.int64)
    return sf_mma[idx]


def assert_quant_equal(q, o, rows=None):
    """q: NVFP4Tensor from the GPU; o: (codes, sf_rowmajor, scale) from the
    oracle for `rows` of Q (all rows if None).  Bit-exact comparison."""
    codes, sf, scale = o
    g_codes = q.codes.cpu().numpy()
    g_sf = q.sf.cpu().numpy()
    g_scale = q.tensor_scale.cpu().numpy()[0]
    assert g_scale.view(np.uint32) == np.float32(scale).view(np.uint32), (g_scale, scale)
    kb = q.k // 16
    if rows is None:
        rows = np.arange(q.rows)
    if len(rows) == 0:
        return
    gc = g_codes[rows]
    if not np.array_equal(gc, codes):
        bad = np.argwhere(gc != codes)
        r, c = bad[0]
        raise AssertionError("codes differ at %d places; first row %d byte %d: gpu %02x oracle %02x"
                             % (len(bad), rows[r], c, gc[r, c], codes[r, c]))
    if q.sf_layout == nv.NVFP4_SF_MMA:
        gs = sf_rows_from_mma(g_sf, rows, kb, q.k)
    else:
        gs = g_sf[: q.rows * kb].reshape(q.rows, kb)[rows]
    if not np.array_equal(gs, sf):
        bad = np.argwhere(gs != sf)
        r, c = bad[0]
        raise AssertionError("scales differ at %d places; first row %d block %d: gpu %02x oracle %02x"
                             % (len(bad), rows[r], c, gs[r, c], sf[r, c]))


def rel_err(got, ref):
    """max |got - ref| / max(|ref|, 1e-3 * max|ref|)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    floor = 1e-3 * max(np.abs(ref).max(), 1e-300)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


def bf16_within_one_ulp(got_bf16, ref):
    """|got - ref| <= one BF16 ulp at max(|ref|, 1e-3 * max|ref|)."""
    got = np.asarray(got_bf16, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.maximum(np.abs(ref), 1e-3 * max(np.abs(ref).max(), 1e-300))
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    return bool(np.all(np.abs(got - ref) <= ulp))


def to_dev(t):
    return t.to(DEV)


def quant_pair(x_cpu, **mode):
    """GPU and oracle quantisation of the same BF16 tensor."""
    g, o = cfgs(**mode)
    q = nv.nvfp4_quantize(to_dev(x_cpu), g)
    return q, oracle.quantize(syn.as_u16(x_cpu), o)
