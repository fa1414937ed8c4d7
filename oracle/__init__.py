"""NVFP4 oracle -- TEST INFRASTRUCTURE ONLY.

A ctypes front end over the plain-C oracle in ``oracle.c``.  Only the test
suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the GPU library never does, and shares no code with it.
Inputs are numpy arrays (BF16 as ``uint16`` bit patterns); outputs are numpy
arrays.  Every function maps one-to-one onto a C function in ``oracle.c``,
whose comments cite the passage each step follows.
"""
import ctypes
import os

import numpy as np

from .build import build as _build

_LIB = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_NONFINITE = 0, 1, 2, 6


class OracleError(RuntimeError):
    def __init__(self, status):
        super().__init__("oracle status %d" % status)
        self.status = status


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("block", ctypes.c_int32),
        ("rounding", ctypes.c_int32),
        ("rht", ctypes.c_int32),
        ("transpose", ctypes.c_int32),
        ("rht_seed", ctypes.c_uint64),
        ("sr_seed", ctypes.c_uint64),
        ("sr_offset", ctypes.c_uint64),
    ]


class _NsTrace(ctypes.Structure):
    _fields_ = [("qx", ctypes.c_float), ("qa", ctypes.c_float), ("qb", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("xc", "a", "ac", "a2", "b", "bc", "bx")]


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(_build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode_rne.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode_rne.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode_sr.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_rht_signs.restype = None
        lib.oracle_rht_signs.argtypes = [ctypes.c_uint64, P]
        lib.oracle_rht16.restype = None
        lib.oracle_rht16.argtypes = [P, P]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_quantize.argtypes = [P, I64, I64, I64, ctypes.POINTER(_Cfg), P, P, P]
        lib.oracle_quantize_rows.restype = ctypes.c_int
        lib.oracle_quantize_rows.argtypes = [P, I64, I64, I64, ctypes.POINTER(_Cfg), I64, I64, P, P, P]
        lib.oracle_quantize_given_amax.restype = ctypes.c_int
        lib.oracle_quantize_given_amax.argtypes = [P, I64, I64, I64, ctypes.POINTER(_Cfg), ctypes.c_float, P, P, P]
        lib.oracle_amax.restype = ctypes.c_int
        lib.oracle_amax.argtypes = [P, I64, I64, I64, ctypes.POINTER(_Cfg), P]
        lib.oracle_sf_mma_offset.restype = I64
        lib.oracle_sf_mma_offset.argtypes = [I64, I64, I64]
        lib.oracle_sf_mma_bytes.restype = I64
        lib.oracle_sf_mma_bytes.argtypes = [I64, I64]
        lib.oracle_sf_to_mma.restype = None
        lib.oracle_sf_to_mma.argtypes = [P, I64, I64, P]
        lib.oracle_dequantize.restype = None
        lib.oracle_dequantize.argtypes = [P, P, ctypes.c_float, I64, I64, P]
        lib.oracle_gemm_f64.restype = None
        lib.oracle_gemm_f64.argtypes = [P, P, ctypes.c_float, P, P, ctypes.c_float, I64, I64, I64, P]
        lib.oracle_gemm_f64_sampled.restype = None
        lib.oracle_gemm_f64_sampled.argtypes = [P, P, ctypes.c_float, P, P, ctypes.c_float,
                                                I64, P, P, I64, P]
        U64 = ctypes.c_uint64
        lib.oracle_rht16_inverse.restype = None
        lib.oracle_rht16_inverse.argtypes = [P, P]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_qadamw_m_encode.restype = ctypes.c_int
        lib.oracle_qadamw_m_encode.argtypes = [P, I64, I64, U64, U64, U64, P, P, P]
        lib.oracle_qadamw_m_decode.restype = None
        lib.oracle_qadamw_m_decode.argtypes = [P, P, ctypes.c_float, I64, I64, U64, P]
        lib.oracle_qadamw_v_encode.restype = ctypes.c_int
        lib.oracle_qadamw_v_encode.argtypes = [P, I64, I64, U64, P, P, P, P]
        lib.oracle_qadamw_v_decode.restype = None
        lib.oracle_qadamw_v_decode.argtypes = [P, P, ctypes.c_float, P, I64, I64, U64, P]
        lib.oracle_lora_forward.restype = None
        lib.oracle_lora_forward.argtypes = [P, P, ctypes.c_float, P, P, ctypes.c_float, P, P, P, ctypes.c_double,
                                            I64, I64, I64, I64, P]
        lib.oracle_lora_down.restype = None
        lib.oracle_lora_down.argtypes = [P, P, I64, I64, I64, P, P]
        lib.oracle_lora_forward_sampled.restype = None
        lib.oracle_lora_forward_sampled.argtypes = [P, P, ctypes.c_float, P, P, ctypes.c_float, P, P, P,
                                                    ctypes.c_double, I64, I64, P, P, I64, P]
        lib.oracle_bf16_rne_f64.restype = ctypes.c_uint16
        lib.oracle_bf16_rne_f64.argtypes = [ctypes.c_double]
        lib.oracle_axpby_bf16.restype = None
        lib.oracle_axpby_bf16.argtypes = [P, P, I64, ctypes.c_float, ctypes.c_float, P]
        lib.oracle_ns_step.restype = ctypes.c_int
        lib.oracle_ns_step.argtypes = [P, I64, I64, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_double,
                                       P, ctypes.POINTER(_NsTrace)]
        lib.oracle_abs_percentile_bf16.restype = ctypes.c_float
        lib.oracle_abs_percentile_bf16.argtypes = [P, I64, ctypes.c_double]
        lib.oracle_clip_bf16.restype = None
        lib.oracle_clip_bf16.argtypes = [P, I64, ctypes.c_float, P]
        _LIB = lib
    return _LIB


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def make_cfg(block=0, rounding=0, rht=0, transpose=0, rht_seed=0, sr_seed=0, sr_offset=0):
    return dict(block=block, rounding=rounding, rht=rht, transpose=transpose,
                rht_seed=rht_seed, sr_seed=sr_seed, sr_offset=sr_offset)


def _cfg(cfg):
    c = make_cfg(**(cfg or {}))
    return _Cfg(c["block"], c["rounding"], c["rht"], c["transpose"],
                c["rht_seed"], c["sr_seed"], c["sr_offset"])


# --- codecs -----------------------------------------------------------------
def e2m1_value(code):
    return _lib().oracle_e2m1_value(int(code))


def e4m3_value(byte):
    return _lib().oracle_e4m3_value(int(byte))


def e4m3_encode(t):
    return _lib().oracle_e4m3_encode(float(t))


def e2m1_encode_rne(v):
    return _lib().oracle_e2m1_encode_rne(float(v))


def e2m1_encode_sr(v, r):
    return _lib().oracle_e2m1_encode_sr(float(v), int(r) & 0xFFFFFFFF)


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def rht_signs(seed):
    sigma = np.zeros(16, dtype=np.float32)
    _lib().oracle_rht_signs(int(seed), _ptr(sigma))
    return sigma


def rht16(v, sigma):
    out = np.ascontiguousarray(v, dtype=np.float32).copy()
    s = np.ascontiguousarray(sigma, dtype=np.float32)
    _lib().oracle_rht16(_ptr(out), _ptr(s))
    return out


# --- quantisation -----------------------------------------------------------
def quantize(x_u16, cfg=None):
    """x_u16: uint16 [rows, cols] BF16 bit patterns (row-major, may be a
    strided view along rows).  Returns (codes [qr, qk/2] u8, sf [qr, qk/16]
    u8 row-major, tensor_scale float32)."""
    x = np.asarray(x_u16)
    assert x.dtype == np.uint16 and x.ndim == 2
    if x.strides[1] != 2:
        x = np.ascontiguousarray(x)
    rows, cols = x.shape
    ld = x.strides[0] // 2 if rows > 1 else cols
    c = _cfg(cfg)
    qr, qk = (cols, rows) if c.transpose else (rows, cols)
    codes = np.zeros((qr, max(qk // 2, 0)), dtype=np.uint8)
    sf = np.zeros((qr, max(qk // 16, 0)), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    st = _lib().oracle_quantize(_ptr(x), rows, cols, ld, ctypes.byref(c), _ptr(codes), _ptr(sf), _ptr(ts))
    if st != OK:
        raise OracleError(st)
    return codes, sf, ts[0]


def quantize_rows(x_u16, cfg, row_begin, row_end):
    """Encode only rows [row_begin, row_end) of Q; the tensor scale is that
    of the whole operand."""
    x = np.ascontiguousarray(x_u16)
    rows, cols = x.shape
    c = _cfg(cfg)
    qr, qk = (cols, rows) if c.transpose else (rows, cols)
    n = row_end - row_begin
    codes = np.zeros((n, qk // 2), dtype=np.uint8)
    sf = np.zeros((n, qk // 16), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    st = _lib().oracle_quantize_rows(_ptr(x), rows, cols, cols, ctypes.byref(c), int(row_begin), int(row_end),
                                     _ptr(codes), _ptr(sf), _ptr(ts))
    if st != OK:
        raise OracleError(st)
    return codes, sf, ts[0]


def quantize_given_amax(x_u16, cfg, amax_value):
    """Delayed scaling: quantise with the tensor scale amax_value / 2688
    instead of the operand's own amax.  Returns (codes, sf, tensor_scale)."""
    x = np.ascontiguousarray(x_u16)
    assert x.dtype == np.uint16 and x.ndim == 2
    rows, cols = x.shape
    c = _cfg(cfg)
    qr, qk = (cols, rows) if c.transpose else (rows, cols)
    codes = np.zeros((qr, max(qk // 2, 0)), dtype=np.uint8)
    sf = np.zeros((qr, max(qk // 16, 0)), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    st = _lib().oracle_quantize_given_amax(_ptr(x), rows, cols, cols, ctypes.byref(c), float(amax_value),
                                           _ptr(codes), _ptr(sf), _ptr(ts))
    if st != OK:
        raise OracleError(st)
    return codes, sf, ts[0]


def amax(x_u16, cfg=None):
    x = np.ascontiguousarray(x_u16)
    rows, cols = x.shape
    c = _cfg(cfg)
    out = np.zeros(1, dtype=np.float32)
    st = _lib().oracle_amax(_ptr(x), rows, cols, cols, ctypes.byref(c), _ptr(out))
    if st != OK:
        raise OracleError(st)
    return out[0]


def sf_mma_offset(r, kb, qk):
    return _lib().oracle_sf_mma_offset(int(r), int(kb), int(qk))


def sf_mma_bytes(qr, qk):
    return _lib().oracle_sf_mma_bytes(int(qr), int(qk))


def sf_to_mma(sf, qr, qk):
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    out = np.zeros(sf_mma_bytes(qr, qk), dtype=np.uint8)
    _lib().oracle_sf_to_mma(_ptr(sf), int(qr), int(qk), _ptr(out))
    return out


def dequantize(codes, sf, tensor_scale, qr, qk):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    out = np.zeros((qr, qk), dtype=np.float64)
    _lib().oracle_dequantize(_ptr(codes), _ptr(sf), float(tensor_scale), int(qr), int(qk), _ptr(out))
    return out


def gemm_f64(a, b, M, N, K):
    """a, b: (codes, sf_rowmajor, tensor_scale) of A [M, K] and B [N, K]."""
    ac, asf, ascale = a
    bc, bsf, bscale = b
    ac, asf = np.ascontiguousarray(ac), np.ascontiguousarray(asf)
    bc, bsf = np.ascontiguousarray(bc), np.ascontiguousarray(bsf)
    out = np.zeros((M, N), dtype=np.float64)
    _lib().oracle_gemm_f64(_ptr(ac), _ptr(asf), float(ascale), _ptr(bc), _ptr(bsf), float(bscale),
                           int(M), int(N), int(K), _ptr(out))
    return out


def gemm_f64_sampled(a, b, K, m_idx, n_idx):
    ac, asf, ascale = a
    bc, bsf, bscale = b
    ac, asf = np.ascontiguousarray(ac), np.ascontiguousarray(asf)
    bc, bsf = np.ascontiguousarray(bc), np.ascontiguousarray(bsf)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.zeros(mi.shape[0], dtype=np.float64)
    _lib().oracle_gemm_f64_sampled(_ptr(ac), _ptr(asf), float(ascale), _ptr(bc), _ptr(bsf), float(bscale),
                                   int(K), _ptr(mi), _ptr(ni), int(mi.shape[0]), _ptr(out))
    return out


# --- quantised AdamW state codec -------------------------------------------
def rht16_inverse(v, sigma):
    out = np.ascontiguousarray(v, dtype=np.float32).copy()
    s = np.ascontiguousarray(sigma, dtype=np.float32)
    _lib().oracle_rht16_inverse(_ptr(out), _ptr(s))
    return out


def bf16_rne(f):
    return _lib().oracle_bf16_rne(float(f))


def qadamw_m_encode(m, rht_seed, sr_seed, sr_offset=0):
    """m: float32 [rows, cols].  Returns (codes, sf row-major, tensor_scale)."""
    m = np.ascontiguousarray(m, dtype=np.float32)
    rows, cols = m.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    sf = np.zeros((rows, cols // 16), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    st = _lib().oracle_qadamw_m_encode(_ptr(m), rows, cols, int(rht_seed), int(sr_seed), int(sr_offset),
                                       _ptr(codes), _ptr(sf), _ptr(ts))
    if st != OK:
        raise OracleError(st)
    return codes, sf, ts[0]


def qadamw_m_decode(codes, sf, tensor_scale, rows, cols, rht_seed):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    out = np.zeros((rows, cols), dtype=np.float32)
    _lib().oracle_qadamw_m_decode(_ptr(codes), _ptr(sf), float(tensor_scale), int(rows), int(cols), int(rht_seed),
                                  _ptr(out))
    return out


def qadamw_v_encode(v, rht_seed):
    """v: float32 [rows, cols] >= 0.  Returns (codes, sf row-major,
    tensor_scale, tile means [rows/16, cols/16] as uint16 BF16 bits)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows, cols = v.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    sf = np.zeros((rows, cols // 16), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    mu = np.zeros((max(rows // 16, 0), max(cols // 16, 0)), dtype=np.uint16)
    st = _lib().oracle_qadamw_v_encode(_ptr(v), rows, cols, int(rht_seed), _ptr(codes), _ptr(sf), _ptr(ts), _ptr(mu))
    if st != OK:
        raise OracleError(st)
    return codes, sf, ts[0], mu


def qadamw_v_decode(codes, sf, tensor_scale, tile_mean, rows, cols, rht_seed):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    mu = np.ascontiguousarray(tile_mean, dtype=np.uint16)
    out = np.zeros((rows, cols), dtype=np.float32)
    _lib().oracle_qadamw_v_decode(_ptr(codes), _ptr(sf), float(tensor_scale), _ptr(mu), int(rows), int(cols),
                                  int(rht_seed), _ptr(out))
    return out


# --- LoRA-SVD projection -----------------------------------------------------
def lora_forward(xq, wq, x_u16, l1_u16, l2_u16, beta):
    """xq, wq: (codes, sf row-major, tensor_scale) of X [T, din] and W_res
    [dout, din]; x, l1 [r, din], l2 [dout, r] as BF16 bit patterns.  Returns
    Y [T, dout] in FP64."""
    xc, xsf, xs = xq
    wc, wsf, ws = wq
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    l1 = np.ascontiguousarray(l1_u16, dtype=np.uint16)
    l2 = np.ascontiguousarray(l2_u16, dtype=np.uint16)
    T, din = x.shape
    dout, r = l2.shape
    out = np.zeros((T, dout), dtype=np.float64)
    xc, xsf, wc, wsf = (np.ascontiguousarray(a) for a in (xc, xsf, wc, wsf))
    _lib().oracle_lora_forward(_ptr(xc), _ptr(xsf), float(xs), _ptr(wc), _ptr(wsf), float(ws), _ptr(x), _ptr(l1),
                               _ptr(l2), float(beta), int(T), int(din), int(dout), int(r), _ptr(out))
    return out


def lora_down(x_u16, l1_u16):
    """U = BF16(X L1^T) [T, r] (uint16 bits) and the exact FP64 sums it rounds."""
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    l1 = np.ascontiguousarray(l1_u16, dtype=np.uint16)
    T, din = x.shape
    r = l1.shape[0]
    u = np.zeros((T, r), dtype=np.uint16)
    ue = np.zeros((T, r), dtype=np.float64)
    _lib().oracle_lora_down(_ptr(x), _ptr(l1), int(T), int(din), int(r), _ptr(u), _ptr(ue))
    return u, ue


def lora_forward_sampled(xq, wq, x_u16, l1_u16, l2_u16, beta, t_idx, n_idx):
    """Y of lora_forward at the coordinates (t_idx[i], n_idx[i]) only."""
    xc, xsf, xs = xq
    wc, wsf, ws = wq
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    l1 = np.ascontiguousarray(l1_u16, dtype=np.uint16)
    l2 = np.ascontiguousarray(l2_u16, dtype=np.uint16)
    din = x.shape[1]
    r = l2.shape[1]
    ti = np.ascontiguousarray(t_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.zeros(ti.size, dtype=np.float64)
    xc, xsf, wc, wsf = (np.ascontiguousarray(a) for a in (xc, xsf, wc, wsf))
    _lib().oracle_lora_forward_sampled(_ptr(xc), _ptr(xsf), float(xs), _ptr(wc), _ptr(wsf), float(ws), _ptr(x),
                                       _ptr(l1), _ptr(l2), float(beta), int(din), int(r), _ptr(ti), _ptr(ni),
                                       int(ti.size), _ptr(out))
    return out


# --- Newton-Schulz step with NVFP4 products ----------------------------------
def bf16_rne_f64(d):
    return _lib().oracle_bf16_rne_f64(float(d))


def axpby_bf16(x_u16, y_u16, a, b):
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    y = np.ascontiguousarray(y_u16, dtype=np.uint16)
    out = np.zeros_like(x)
    _lib().oracle_axpby_bf16(_ptr(x), _ptr(y), int(x.size), float(a), float(b), _ptr(out))
    return out


def ns_step(x_u16, a, b, c, p=99.0):
    """One Newton-Schulz step (see oracle.c).  Returns (X' as uint16 BF16 bits,
    trace dict with the clip thresholds qx, qa, qb and the BF16 intermediates
    xc, a, ac, a2, b, bc, bx)."""
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    m, n = x.shape
    out = np.zeros_like(x)
    bufs = {k: np.zeros((m, n) if k in ("xc", "bx") else (m, m), dtype=np.uint16)
            for k in ("xc", "a", "ac", "a2", "b", "bc", "bx")}
    tr = _NsTrace(0.0, 0.0, 0.0, *[bufs[k].ctypes.data for k in ("xc", "a", "ac", "a2", "b", "bc", "bx")])
    st = _lib().oracle_ns_step(_ptr(x), int(m), int(n), float(a), float(b), float(c), float(p), _ptr(out),
                               ctypes.byref(tr))
    if st != OK:
        raise OracleError(st)
    trace = dict(bufs)
    trace.update(qx=np.float32(tr.qx), qa=np.float32(tr.qa), qb=np.float32(tr.qb))
    return out, trace


# --- p99 clipping ---------------------------------------------------------
def abs_percentile_bf16(x_u16, p=99.0):
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    return np.float32(_lib().oracle_abs_percentile_bf16(_ptr(x), int(x.size), float(p)))


def clip_bf16(x_u16, c):
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    out = np.zeros_like(x)
    _lib().oracle_clip_bf16(_ptr(x), int(x.size), float(c), _ptr(out))
    return out
