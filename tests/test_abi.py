"""The C ABI boundary without a GPU: the library loads, exports every symbol
that include/nvfp4.h declares, and rejects bad arguments before launching
anything."""
import ctypes
import os
import re

import pytest

import block_scaled_gemm_nvfp4_gb300 as nv
from block_scaled_gemm_nvfp4_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return nv.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 14
    assert sorted(nv.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert nv.nvfp4_status_string(s)
    assert nv.nvfp4_version() >= 100


def test_sizes(lib):
    assert nv.nvfp4_codes_bytes(4, 32) == 64
    assert nv.nvfp4_sf_bytes(4, 32, nv.NVFP4_SF_ROWMAJOR) == 8
    assert nv.nvfp4_sf_bytes(4, 32, nv.NVFP4_SF_MMA) == 512
    assert nv.nvfp4_sf_bytes(129, 320, nv.NVFP4_SF_MMA) == 2 * 5 * 512


def _q(lib, x=8192, rows=64, cols=64, ldx=64, cfg=None, codes=8192, sf=8192, scale=8192, ws=8192, wsb=1 << 20):
    c = cfg if cfg is not None else nv.quant_cfg()
    P = ctypes.c_void_p
    return lib.nvfp4_quantize(P(x), rows, cols, ldx, ctypes.byref(c), P(codes), P(sf), P(scale), P(ws), wsb,
                              P(0))


def test_quantize_validation(lib):
    # fake, aligned, never dereferenced addresses: every case fails before launch
    assert _q(lib, cfg=nv.quant_cfg(block=7)) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, cfg=nv.quant_cfg(rounding=3)) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, cfg=nv.quant_cfg(sf_layout=9)) == nv.NVFP4_ERR_INVALID_ARG
    bad = nv.quant_cfg()
    bad.reserved = 1
    assert _q(lib, cfg=bad) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, cols=40, ldx=40) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert _q(lib, rows=24, cfg=nv.quant_cfg(block=1)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert _q(lib, rows=40, cfg=nv.quant_cfg(transpose=1)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert _q(lib, ldx=32) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, x=8194) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, ldx=68) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, x=0) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, scale=0) == nv.NVFP4_ERR_INVALID_ARG
    assert _q(lib, ws=0) == nv.NVFP4_ERR_WORKSPACE
    assert _q(lib, wsb=100) == nv.NVFP4_ERR_WORKSPACE
    assert lib.nvfp4_quantize(ctypes.c_void_p(8192), 64, 64, 64, None, ctypes.c_void_p(8192),
                              ctypes.c_void_p(8192), ctypes.c_void_p(8192), ctypes.c_void_p(8192), 1 << 20,
                              ctypes.c_void_p(0)) == nv.NVFP4_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert lib.nvfp4_quantize_workspace_size(64, 64, ctypes.byref(nv.quant_cfg()), ctypes.byref(n)) == 0
    assert n.value >= 256


def _t(codes=8192, sf=8192, scale=8192, rows=64, k=64, layout=nv.NVFP4_SF_MMA):
    return nv._Tensor(codes, sf, scale, rows, k, layout, 0)


def test_gemm_validation(lib):
    P = ctypes.c_void_p

    def g(a, b, dt=0, d=8192, ldd=64, ws=8192, wsb=4096):
        return lib.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), dt, P(d), ldd, P(ws), wsb, P(0))

    assert g(_t(k=48), _t(k=48)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE      # K % 32
    assert g(_t(k=64), _t(k=96)) == nv.NVFP4_ERR_INVALID_ARG            # K mismatch
    assert g(_t(layout=0), _t()) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE      # scales not in MMA layout
    assert g(_t(), _t(), dt=5) == nv.NVFP4_ERR_INVALID_ARG
    assert g(_t(), _t(), d=0) == nv.NVFP4_ERR_INVALID_ARG
    assert g(_t(), _t(rows=100), ldd=64) == nv.NVFP4_ERR_INVALID_ARG    # ldd < N
    assert g(_t(codes=8200), _t()) == nv.NVFP4_ERR_INVALID_ARG          # codes not 16-byte aligned
    assert g(_t(), _t(), ws=0) == nv.NVFP4_ERR_WORKSPACE
    assert g(_t(), _t(), wsb=16) == nv.NVFP4_ERR_WORKSPACE
    assert g(_t(scale=0), _t()) == nv.NVFP4_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert lib.nvfp4_gemm_workspace_size(128, 128, 80, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm_workspace_size(128, 128, 128, ctypes.byref(n)) == 0 and n.value >= 4
    plan = (ctypes.c_int64 * 8)(*range(1, 9))
    assert lib.nvfp4_gemm_plan(256, 256, 1024, 1 << 20, None) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_gemm_plan(-1, 256, 1024, 1 << 20, plan) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_gemm_plan(256, 256, 1000, 1 << 20, plan) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    # an empty output has an empty schedule (no device needed)
    assert lib.nvfp4_gemm_plan(0, 256, 1024, 1 << 20, plan) == 0 and list(plan) == [0] * 8


def test_linear_validation(lib):
    P = ctypes.c_void_p
    n = ctypes.c_size_t(0)
    assert lib.nvfp4_linear_workspace_size(9, 64, 64, 64, ctypes.byref(n)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_linear_workspace_size(0, 64, 48, 64, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_linear_workspace_size(2, 48, 64, 64, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_linear_workspace_size(2, 64, 64, 64, ctypes.byref(n)) == 0
    need = n.value
    args = (P(8192), P(8192), 64, 64, 64, None, None, 0, P(8192))
    assert lib.nvfp4_linear_wgrad(*args, P(8192), need - 1, P(0)) == nv.NVFP4_ERR_WORKSPACE
    assert lib.nvfp4_linear_fprop(P(0), P(8192), 64, 64, 64, None, None, 0, P(8192), P(8192), 1 << 24,
                                  P(0)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_linear_dgrad(P(8192), P(8192), 64, 64, 64, None, None, 3, P(8192), P(8192), 1 << 24,
                                  P(0)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_check_device_status(P(0), P(0)) == nv.NVFP4_ERR_INVALID_ARG


def test_given_amax_validation(lib):
    P = ctypes.c_void_p
    c = nv.quant_cfg()

    def q(amax=8192, cfg=c, cols=64, ws=8192, wsb=1 << 20):
        return lib.nvfp4_quantize_given_amax(P(8192), 64, cols, cols, ctypes.byref(cfg), P(amax), P(8192), P(8192),
                                             P(8192), P(ws), wsb, P(0))

    assert q(amax=0) == nv.NVFP4_ERR_INVALID_ARG
    assert q(cfg=nv.quant_cfg(block=7)) == nv.NVFP4_ERR_INVALID_ARG
    assert q(cols=40) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert q(ws=0) == nv.NVFP4_ERR_WORKSPACE
    assert q(wsb=64) == nv.NVFP4_ERR_WORKSPACE
    assert q(ws=8192 + 64) == nv.NVFP4_ERR_INVALID_ARG  # workspace not 256-byte aligned


def test_gemm_quantize_validation(lib):
    P = ctypes.c_void_p

    def out(amax_in=8192, amax_out=0, codes=8192, sf=8192, scale=8192, layout=nv.NVFP4_SF_MMA, reserved=0):
        return nv._QuantOut(amax_in, amax_out, codes, sf, scale, layout, reserved)

    def g(a=None, b=None, q=None, d=8192, ldd=64, ws=8192, wsb=4096):
        a = a if a is not None else _t()
        b = b if b is not None else _t()
        qq = ctypes.byref(q) if q is not None else None
        return lib.nvfp4_gemm_quantize(ctypes.byref(a), ctypes.byref(b), P(d), ldd, qq, P(ws), wsb, P(0))

    assert g(q=None) == nv.NVFP4_ERR_INVALID_ARG
    assert g(q=out(amax_in=0)) == nv.NVFP4_ERR_INVALID_ARG
    assert g(q=out(scale=0)) == nv.NVFP4_ERR_INVALID_ARG
    assert g(q=out(reserved=1)) == nv.NVFP4_ERR_INVALID_ARG
    assert g(q=out(layout=4)) == nv.NVFP4_ERR_INVALID_ARG
    assert g(b=_t(rows=48), q=out(), ldd=64) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE   # N % 32
    assert g(a=_t(k=0), b=_t(k=0), q=out()) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE   # K = 0
    assert g(a=_t(k=64), b=_t(k=96), q=out()) == nv.NVFP4_ERR_INVALID_ARG
    assert g(q=out(codes=8200)) == nv.NVFP4_ERR_INVALID_ARG                    # codes not 16-byte aligned
    assert g(q=out(sf=8200)) == nv.NVFP4_ERR_INVALID_ARG                       # MMA scales not 16-byte aligned
    assert g(q=out(amax_out=8194)) == nv.NVFP4_ERR_INVALID_ARG                 # amax_out not 4-byte aligned
    assert g(q=out(), ldd=32) == nv.NVFP4_ERR_INVALID_ARG                      # ldd < N with D stored
    assert g(q=out(), ws=0) == nv.NVFP4_ERR_WORKSPACE
    assert g(q=out(), wsb=16) == nv.NVFP4_ERR_WORKSPACE


def test_qadamw_validation(lib):
    P = ctypes.c_void_p
    n = ctypes.c_size_t(0)
    assert lib.nvfp4_qadamw_workspace_size(ctypes.byref(n)) == 0 and n.value >= 256
    assert lib.nvfp4_qadamw_workspace_size(None) == nv.NVFP4_ERR_INVALID_ARG

    def m_enc(m=8192, rows=32, cols=64, codes=8192, sf=8192, scale=8192, ws=8192, wsb=1 << 12):
        return lib.nvfp4_qadamw_m_encode(P(m), rows, cols, 1, 2, 3, P(codes), P(sf), P(scale), P(ws), wsb, P(0))

    assert m_enc(cols=40) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert m_enc(rows=-1) == nv.NVFP4_ERR_INVALID_ARG
    assert m_enc(m=0) == nv.NVFP4_ERR_INVALID_ARG
    assert m_enc(m=8196) == nv.NVFP4_ERR_INVALID_ARG          # state not 16-byte aligned
    assert m_enc(codes=8196) == nv.NVFP4_ERR_INVALID_ARG      # codes not 8-byte aligned
    assert m_enc(scale=0) == nv.NVFP4_ERR_INVALID_ARG
    assert m_enc(ws=0) == nv.NVFP4_ERR_WORKSPACE
    assert m_enc(wsb=8) == nv.NVFP4_ERR_WORKSPACE

    def v_enc(rows=32, cols=64, mean=8192, ws=8192):
        return lib.nvfp4_qadamw_v_encode(P(8192), rows, cols, 1, P(8192), P(8192), P(8192), P(mean), P(ws),
                                         1 << 12, P(0))

    assert v_enc(rows=24) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE  # 16x16 tiles
    assert v_enc(mean=0) == nv.NVFP4_ERR_INVALID_ARG
    assert v_enc(mean=8193) == nv.NVFP4_ERR_INVALID_ARG      # BF16 means need 2-byte alignment
    assert v_enc(ws=0) == nv.NVFP4_ERR_WORKSPACE
    assert lib.nvfp4_qadamw_m_decode(P(8192), P(8192), P(0), 32, 64, 1, P(8192), P(0)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_qadamw_v_decode(P(8192), P(8192), P(8192), P(0), 32, 64, 1, P(8192),
                                     P(0)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_qadamw_v_decode(P(8192), P(8192), P(8192), P(8192), 24, 64, 1, P(8192),
                                     P(0)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE


def test_lora_validation(lib):
    P = ctypes.c_void_p
    n = ctypes.c_size_t(0)
    assert lib.nvfp4_lora_workspace_size(1000, 64, ctypes.byref(n)) == nv.NVFP4_OK
    assert n.value >= 256 + 1000 * 128 * 2
    assert lib.nvfp4_lora_workspace_size(1000, 12, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_lora_workspace_size(1000, 512, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    t = nv._Tensor(8192, 8192, 8192, 64, 64, nv.NVFP4_SF_MMA, 0)
    w_bad_k = nv._Tensor(8192, 8192, 8192, 64, 96, nv.NVFP4_SF_MMA, 0)

    def call(a=t, b=t, r=64, beta=1.0, ws=1 << 20, ldx=64):
        return lib.nvfp4_lora_forward(ctypes.byref(a), ctypes.byref(b), P(8192), ldx, P(8192), P(8192), r,
                                      beta, 0, P(8192), 64, P(8192), P(8192), ws, P(0))

    assert call(b=w_bad_k) == nv.NVFP4_ERR_INVALID_ARG
    assert call(r=20) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert call(beta=float("nan")) == nv.NVFP4_ERR_INVALID_ARG
    assert call(beta=float("inf")) == nv.NVFP4_ERR_INVALID_ARG
    assert call(ws=100) == nv.NVFP4_ERR_WORKSPACE
    assert call(ldx=60) == nv.NVFP4_ERR_INVALID_ARG


def test_ns_validation(lib):
    P = ctypes.c_void_p
    n = ctypes.c_size_t(0)
    assert lib.nvfp4_ns_workspace_size(64, 96, ctypes.byref(n)) == nv.NVFP4_OK and n.value > 6 * 64 * 64
    assert lib.nvfp4_ns_workspace_size(48, 96, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_ns_workspace_size(64, 0, ctypes.byref(n)) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_ns_step(P(8192), 64, 64, 1.0, 0.0, 0.0, 99.0, P(8192), P(8192), 16, P(0)) == \
        nv.NVFP4_ERR_WORKSPACE
    assert lib.nvfp4_ns_step(P(8192), 64, 64, 1.0, 0.0, 0.0, 0.0, P(8192), P(8192), 1 << 30, P(0)) == \
        nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_ns_step(P(8192), 64, 64, 1.0, 0.0, 0.0, 101.0, P(8192), P(8192), 1 << 30, P(0)) == \
        nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_abs_percentile_bf16(P(8192), 100, 99.0, P(8192), P(8192), 16, P(0)) == nv.NVFP4_ERR_WORKSPACE
    assert lib.nvfp4_abs_percentile_bf16(P(8194), 100, 99.0, P(8192), P(8192), 1 << 20, P(0)) == \
        nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_clip_bf16(P(8192), 10, None, P(8192), P(0)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_axpby_bf16(P(8192), P(8200), 10, 1.0, 1.0, P(8192), P(0)) == nv.NVFP4_ERR_INVALID_ARG


def test_mma_rate_validation(lib):
    d = ctypes.c_double()
    for kind, iters in ((-1, 64), (4, 64), (0, 8), (0, (1 << 20) + 1)):
        assert lib.nvfp4_debug_mma_rate(kind, iters, ctypes.byref(d), ctypes.byref(d)) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_debug_mma_rate(0, 64, None, ctypes.byref(d)) == nv.NVFP4_ERR_INVALID_ARG
