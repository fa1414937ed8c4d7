"""libnvfp4: NVFP4 quantisation and block-scaled FP4 GEMM for GB300 (sm_103a).

A thin ctypes binding over the C ABI declared in ``include/nvfp4.h``.  The
Python functions carry the C names and only marshal arguments: device
pointers and sizes from torch tensors, the current CUDA stream, workspaces
allocated with torch.  Every step of the computation runs in the library's
CUDA kernels; if the library is not built, every call raises.
"""
import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libnvfp4.so")

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_UNSUPPORTED_SHAPE = 2
NVFP4_ERR_WORKSPACE = 3
NVFP4_ERR_CUDA = 4
NVFP4_ERR_TIMEOUT = 5
NVFP4_ERR_NONFINITE = 6

NVFP4_BLOCK_1x16, NVFP4_BLOCK_16x16 = 0, 1
NVFP4_ROUND_RNE, NVFP4_ROUND_SR = 0, 1
NVFP4_SF_ROWMAJOR, NVFP4_SF_MMA = 0, 1
NVFP4_OUT_BF16, NVFP4_OUT_F32 = 0, 1
NVFP4_LINEAR_FPROP, NVFP4_LINEAR_DGRAD, NVFP4_LINEAR_WGRAD = 0, 1, 2

# Every exported symbol of include/nvfp4.h.
EXPORTS = [
    "nvfp4_status_string", "nvfp4_version", "nvfp4_codes_bytes", "nvfp4_sf_bytes",
    "nvfp4_quantize_workspace_size", "nvfp4_quantize", "nvfp4_quantize_dual", "nvfp4_quantize_given_amax",
    "nvfp4_quantize_noalloc", "nvfp4_dequantize",
    "nvfp4_gemm_workspace_size", "nvfp4_gemm_plan", "nvfp4_gemm", "nvfp4_gemm_quantize", "nvfp4_linear_workspace_size",
    "nvfp4_linear_fprop", "nvfp4_linear_dgrad", "nvfp4_linear_wgrad",
    "nvfp4_check_device_status", "nvfp4_debug_gemm_skip_load", "nvfp4_debug_quantize_skip_load",
    "nvfp4_qadamw_workspace_size", "nvfp4_qadamw_m_encode", "nvfp4_qadamw_m_decode", "nvfp4_qadamw_v_encode",
    "nvfp4_qadamw_v_decode", "nvfp4_lora_workspace_size", "nvfp4_lora_forward",
    "nvfp4_abs_percentile_workspace_size", "nvfp4_abs_percentile_bf16", "nvfp4_clip_bf16", "nvfp4_axpby_bf16",
    "nvfp4_ns_workspace_size", "nvfp4_ns_step", "nvfp4_debug_mma_rate",
]


class Nvfp4Error(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        msg = nvfp4_status_string(status) if _LIB is not None else "status %d" % status
        super().__init__("%s: %s (status %d)" % (what, msg, status) if what else "%s (status %d)" % (msg, status))


class QuantCfg(ctypes.Structure):
    """nvfp4_quant_cfg."""
    _fields_ = [
        ("block", ctypes.c_int32),
        ("rounding", ctypes.c_int32),
        ("rht", ctypes.c_int32),
        ("sf_layout", ctypes.c_int32),
        ("transpose", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("rht_seed", ctypes.c_uint64),
        ("sr_seed", ctypes.c_uint64),
        ("sr_offset", ctypes.c_uint64),
    ]


def quant_cfg(block=0, rounding=0, rht=0, sf_layout=NVFP4_SF_MMA, transpose=0, rht_seed=0, sr_seed=0,
              sr_offset=0):
    return QuantCfg(block, rounding, rht, sf_layout, transpose, 0, rht_seed, sr_seed, sr_offset)


class _Tensor(ctypes.Structure):
    """nvfp4_tensor."""
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("sf", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("k", ctypes.c_int64),
        ("sf_layout", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class _QuantOut(ctypes.Structure):
    """nvfp4_quant_out."""
    _fields_ = [
        ("amax_in", ctypes.c_void_p),
        ("amax_out", ctypes.c_void_p),
        ("codes", ctypes.c_void_p),
        ("sf", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
        ("sf_layout", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


@dataclass
class NVFP4Tensor:
    """A quantised operand Q [rows, k] held in torch device buffers."""
    codes: torch.Tensor         # uint8 [rows, k/2]
    sf: torch.Tensor            # uint8, row-major [rows, k/16] or the padded MMA layout
    tensor_scale: torch.Tensor  # float32 [1]
    rows: int
    k: int
    sf_layout: int

    def _c(self):
        return _Tensor(self.codes.data_ptr(), self.sf.data_ptr(), self.tensor_scale.data_ptr(),
                       self.rows, self.k, self.sf_layout, 0)


_LIB = None


def lib():
    """Load libnvfp4 (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libnvfp4 is not built (%s missing); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        PSZ = ctypes.POINTER(ctypes.c_size_t)
        PCFG = ctypes.POINTER(QuantCfg)
        PT = ctypes.POINTER(_Tensor)
        sigs = {
            "nvfp4_status_string": (ctypes.c_char_p, [I32]),
            "nvfp4_version": (I32, []),
            "nvfp4_codes_bytes": (SZ, [I64, I64]),
            "nvfp4_sf_bytes": (SZ, [I64, I64, I32]),
            "nvfp4_quantize_workspace_size": (I32, [I64, I64, PCFG, PSZ]),
            "nvfp4_quantize": (I32, [P, I64, I64, I64, PCFG, P, P, P, P, SZ, P]),
            "nvfp4_quantize_dual": (I32, [P, I64, I64, I64, PCFG, P, P, P, PCFG, P, P, P, P, SZ, P]),
            "nvfp4_quantize_given_amax": (I32, [P, I64, I64, I64, PCFG, P, P, P, P, P, SZ, P]),
            "nvfp4_quantize_noalloc": (I32, [P, I64, I64, I64, PCFG, P, P, P, P]),
            "nvfp4_dequantize": (I32, [PT, I32, P, I64, P]),
            "nvfp4_gemm_workspace_size": (I32, [I64, I64, I64, PSZ]),
            "nvfp4_gemm_plan": (I32, [I64, I64, I64, SZ, ctypes.POINTER(ctypes.c_int64)]),
            "nvfp4_gemm": (I32, [PT, PT, I32, P, I64, P, SZ, P]),
            "nvfp4_gemm_quantize": (I32, [PT, PT, P, I64, ctypes.POINTER(_QuantOut), P, SZ, P]),
            "nvfp4_linear_workspace_size": (I32, [I32, I64, I64, I64, PSZ]),
            "nvfp4_linear_fprop": (I32, [P, P, I64, I64, I64, PCFG, PCFG, I32, P, P, SZ, P]),
            "nvfp4_linear_dgrad": (I32, [P, P, I64, I64, I64, PCFG, PCFG, I32, P, P, SZ, P]),
            "nvfp4_linear_wgrad": (I32, [P, P, I64, I64, I64, PCFG, PCFG, I32, P, P, SZ, P]),
            "nvfp4_check_device_status": (I32, [P, P]),
            "nvfp4_debug_gemm_skip_load": (None, [I32]),
            "nvfp4_debug_quantize_skip_load": (None, [I32]),
            "nvfp4_debug_mma_rate": (I32, [I32, I32, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double)]),
            "nvfp4_qadamw_workspace_size": (I32, [PSZ]),
            "nvfp4_qadamw_m_encode": (I32, [P, I64, I64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, P, P, P, P,
                                            SZ, P]),
            "nvfp4_qadamw_m_decode": (I32, [P, P, P, I64, I64, ctypes.c_uint64, P, P]),
            "nvfp4_qadamw_v_encode": (I32, [P, I64, I64, ctypes.c_uint64, P, P, P, P, P, SZ, P]),
            "nvfp4_qadamw_v_decode": (I32, [P, P, P, P, I64, I64, ctypes.c_uint64, P, P]),
            "nvfp4_lora_workspace_size": (I32, [I64, I64, PSZ]),
            "nvfp4_lora_forward": (I32, [PT, PT, P, I64, P, P, I64, ctypes.c_float, I32, P, I64, P, P, SZ, P]),
            "nvfp4_abs_percentile_workspace_size": (I32, [PSZ]),
            "nvfp4_abs_percentile_bf16": (I32, [P, I64, ctypes.c_double, P, P, SZ, P]),
            "nvfp4_clip_bf16": (I32, [P, I64, P, P, P]),
            "nvfp4_axpby_bf16": (I32, [P, P, I64, ctypes.c_float, ctypes.c_float, P, P]),
            "nvfp4_ns_workspace_size": (I32, [I64, I64, PSZ]),
            "nvfp4_ns_step": (I32, [P, I64, I64, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_double, P,
                                    P, SZ, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != NVFP4_OK:
        raise Nvfp4Error(status, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def nvfp4_status_string(status):
    return lib().nvfp4_status_string(int(status)).decode()


def nvfp4_version():
    return lib().nvfp4_version()


def nvfp4_codes_bytes(qr, qk):
    return lib().nvfp4_codes_bytes(qr, qk)


def nvfp4_sf_bytes(qr, qk, sf_layout):
    return lib().nvfp4_sf_bytes(qr, qk, sf_layout)


def _alloc_ws(nbytes, device):
    # The 256-byte header (the status word) must start clear; the scratch
    # after it is always written before it is read.
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def nvfp4_quantize_workspace_size(rows, cols, cfg):
    n = ctypes.c_size_t(0)
    _check(lib().nvfp4_quantize_workspace_size(rows, cols, ctypes.byref(cfg), ctypes.byref(n)),
           "nvfp4_quantize_workspace_size")
    return n.value


def nvfp4_empty(x, cfg):
    """Allocate the outputs of quantising x with cfg."""
    rows, cols = x.shape
    qr, qk = (cols, rows) if cfg.transpose else (rows, cols)
    return NVFP4Tensor(
        codes=torch.empty((qr, qk // 2), dtype=torch.uint8, device=x.device),
        sf=torch.empty(max(nvfp4_sf_bytes(qr, qk, cfg.sf_layout), 1), dtype=torch.uint8, device=x.device),
        tensor_scale=torch.empty(1, dtype=torch.float32, device=x.device),
        rows=qr, k=qk, sf_layout=cfg.sf_layout)


def nvfp4_quantize(x, cfg, out=None, workspace=None, stream=None):
    """x: BF16 CUDA tensor [rows, cols] with unit column stride.  Returns an
    NVFP4Tensor (allocated unless `out` is given)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out is None:
        out = nvfp4_empty(x, cfg)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_quantize_workspace_size(rows, cols, cfg), x.device)
    ldx = x.stride(0) if rows > 1 else cols
    st = lib().nvfp4_quantize(_ptr(x), rows, cols, ldx, ctypes.byref(cfg), _ptr(out.codes), _ptr(out.sf),
                              _ptr(out.tensor_scale), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "nvfp4_quantize")
    return out


def nvfp4_quantize_dual(x, cfg_a, cfg_b, out_a=None, out_b=None, workspace=None, stream=None):
    """Two quantised outputs of one BF16 tensor from one read (see
    include/nvfp4.h).  Returns (out_a, out_b)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out_a is None:
        out_a = nvfp4_empty(x, cfg_a)
    if out_b is None:
        out_b = nvfp4_empty(x, cfg_b)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_quantize_workspace_size(rows, cols, cfg_a), x.device)
    ldx = x.stride(0) if rows > 1 else cols
    st = lib().nvfp4_quantize_dual(_ptr(x), rows, cols, ldx, ctypes.byref(cfg_a), _ptr(out_a.codes),
                                   _ptr(out_a.sf), _ptr(out_a.tensor_scale), ctypes.byref(cfg_b),
                                   _ptr(out_b.codes), _ptr(out_b.sf), _ptr(out_b.tensor_scale), _ptr(workspace),
                                   workspace.numel(), _stream(stream))
    _check(st, "nvfp4_quantize_dual")
    return out_a, out_b


def nvfp4_quantize_given_amax(x, cfg, amax, out=None, workspace=None, stream=None):
    """Delayed scaling (see include/nvfp4.h): quantise x with the tensor
    scale amax[0] / 2688, amax a float32 CUDA tensor; one read of x."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert amax.dtype == torch.float32 and amax.is_cuda
    rows, cols = x.shape
    if out is None:
        out = nvfp4_empty(x, cfg)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_quantize_workspace_size(rows, cols, cfg), x.device)
    ldx = x.stride(0) if rows > 1 else cols
    st = lib().nvfp4_quantize_given_amax(_ptr(x), rows, cols, ldx, ctypes.byref(cfg), _ptr(amax), _ptr(out.codes),
                                         _ptr(out.sf), _ptr(out.tensor_scale), _ptr(workspace), workspace.numel(),
                                         _stream(stream))
    _check(st, "nvfp4_quantize_given_amax")
    return out


def nvfp4_quantize_noalloc(x, cfg, out, stream=None):
    """Scratch-free quantisation (see include/nvfp4.h): `out` is a
    preallocated NVFP4Tensor; the library allocates nothing."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    ldx = x.stride(0) if rows > 1 else cols
    st = lib().nvfp4_quantize_noalloc(_ptr(x), rows, cols, ldx, ctypes.byref(cfg), _ptr(out.codes), _ptr(out.sf),
                                      _ptr(out.tensor_scale), _stream(stream))
    _check(st, "nvfp4_quantize_noalloc")
    return out


def nvfp4_dequantize(q, out_dtype=NVFP4_OUT_F32, out=None, stream=None):
    if out is None:
        dt = torch.float32 if out_dtype == NVFP4_OUT_F32 else torch.bfloat16
        out = torch.empty((q.rows, q.k), dtype=dt, device=q.codes.device)
    t = q._c()
    st = lib().nvfp4_dequantize(ctypes.byref(t), out_dtype, _ptr(out), out.stride(0) if q.rows > 1 else q.k,
                                _stream(stream))
    _check(st, "nvfp4_dequantize")
    return out


def nvfp4_gemm_workspace_size(M, N, K):
    n = ctypes.c_size_t(0)
    _check(lib().nvfp4_gemm_workspace_size(M, N, K, ctypes.byref(n)), "nvfp4_gemm_workspace_size")
    return n.value


GEMM_PLAN_KEYS = ("pair", "ctas", "units", "split_k", "kb_per_split", "tail_tiles", "tail_split", "tail_kb")


def nvfp4_gemm_plan(M, N, K, workspace_bytes=None):
    """The schedule nvfp4_gemm uses for this shape with a workspace of that
    many bytes (default: nvfp4_gemm_workspace_size), as a dict."""
    if workspace_bytes is None:
        workspace_bytes = nvfp4_gemm_workspace_size(M, N, K)
    out = (ctypes.c_int64 * 8)()
    _check(lib().nvfp4_gemm_plan(M, N, K, workspace_bytes, out), "nvfp4_gemm_plan")
    return dict(zip(GEMM_PLAN_KEYS, (int(v) for v in out)))


def nvfp4_gemm(a, b, out_dtype=NVFP4_OUT_BF16, d=None, workspace=None, stream=None):
    """D [a.rows, b.rows] = A * B^T on NVFP4 operands."""
    if d is None:
        dt = torch.float32 if out_dtype == NVFP4_OUT_F32 else torch.bfloat16
        d = torch.empty((a.rows, b.rows), dtype=dt, device=a.codes.device)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_gemm_workspace_size(a.rows, b.rows, a.k), a.codes.device)
    ta, tb = a._c(), b._c()
    ldd = d.stride(0) if d.dim() == 2 and d.shape[0] > 1 else b.rows
    st = lib().nvfp4_gemm(ctypes.byref(ta), ctypes.byref(tb), out_dtype, _ptr(d), ldd, _ptr(workspace),
                          workspace.numel(), _stream(stream))
    _check(st, "nvfp4_gemm")
    return d


def nvfp4_gemm_quantize(a, b, amax_in, sf_layout=NVFP4_SF_MMA, d=None, store_d=True, amax_out=None, out=None,
                        workspace=None, stream=None):
    """D [a.rows, b.rows] = A * B^T (BF16) and its NVFP4 quantisation along N
    (1x16, round to nearest even) under the tensor scale amax_in[0] / 2688,
    from the GEMM's epilogue (see include/nvfp4.h).  amax_out, if given,
    receives max |D|.  Returns (d or None, NVFP4Tensor)."""
    M, N = a.rows, b.rows
    dev = a.codes.device
    if d is None and store_d:
        d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if out is None:
        out = NVFP4Tensor(codes=torch.empty((M, N // 2), dtype=torch.uint8, device=dev),
                          sf=torch.empty(max(nvfp4_sf_bytes(M, N, sf_layout), 1), dtype=torch.uint8, device=dev),
                          tensor_scale=torch.empty(1, dtype=torch.float32, device=dev),
                          rows=M, k=N, sf_layout=sf_layout)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_gemm_workspace_size(M, N, a.k), dev)
    ta, tb = a._c(), b._c()
    q = _QuantOut(amax_in.data_ptr(), amax_out.data_ptr() if amax_out is not None else None, out.codes.data_ptr(),
                  out.sf.data_ptr(), out.tensor_scale.data_ptr(), out.sf_layout, 0)
    ldd = d.stride(0) if d is not None and d.shape[0] > 1 else N
    st = lib().nvfp4_gemm_quantize(ctypes.byref(ta), ctypes.byref(tb), _ptr(d), ldd, ctypes.byref(q),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "nvfp4_gemm_quantize")
    return d, out


def nvfp4_linear_workspace_size(op, tokens, din, dout):
    n = ctypes.c_size_t(0)
    _check(lib().nvfp4_linear_workspace_size(op, tokens, din, dout, ctypes.byref(n)),
           "nvfp4_linear_workspace_size")
    return n.value


def _linear(fn, op, a, b, tokens, din, dout, cfg_a, cfg_b, out_dtype, out, out_shape, workspace, stream):
    dt = torch.float32 if out_dtype == NVFP4_OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty(out_shape, dtype=dt, device=a.device)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_linear_workspace_size(op, tokens, din, dout), a.device)
    ca = ctypes.byref(cfg_a) if cfg_a is not None else None
    cb = ctypes.byref(cfg_b) if cfg_b is not None else None
    st = fn(_ptr(a), _ptr(b), tokens, din, dout, ca, cb, out_dtype, _ptr(out), _ptr(workspace), workspace.numel(),
            _stream(stream))
    _check(st, fn.__name__)
    return out


def nvfp4_linear_fprop(x, w, cfg_x=None, cfg_w=None, out_dtype=NVFP4_OUT_BF16, y=None, workspace=None,
                       stream=None):
    """Y [T, dout] = Q(X) Q(W)^T for X [T, din], W [dout, din] (BF16)."""
    T, din = x.shape
    dout = w.shape[0]
    return _linear(lib().nvfp4_linear_fprop, NVFP4_LINEAR_FPROP, x, w, T, din, dout, cfg_x, cfg_w, out_dtype, y,
                   (T, dout), workspace, stream)


def nvfp4_linear_dgrad(dy, w, cfg_dy=None, cfg_w=None, out_dtype=NVFP4_OUT_BF16, dx=None, workspace=None,
                       stream=None):
    """dX [T, din] = Q(dY) Q(W^T)^T for dY [T, dout], W [dout, din]."""
    T, dout = dy.shape
    din = w.shape[1]
    return _linear(lib().nvfp4_linear_dgrad, NVFP4_LINEAR_DGRAD, dy, w, T, din, dout, cfg_dy, cfg_w, out_dtype,
                   dx, (T, din), workspace, stream)


def nvfp4_linear_wgrad(dy, x, cfg_dy=None, cfg_x=None, out_dtype=NVFP4_OUT_BF16, dw=None, workspace=None,
                       stream=None):
    """dW [dout, din] = Q(dY^T) Q(X^T)^T for dY [T, dout], X [T, din]."""
    T, dout = dy.shape
    din = x.shape[1]
    return _linear(lib().nvfp4_linear_wgrad, NVFP4_LINEAR_WGRAD, dy, x, T, din, dout, cfg_dy, cfg_x, out_dtype,
                   dw, (dout, din), workspace, stream)


NVFP4_DEFAULT_RHT_SEED = 0x5EEDC0DE0F4


def nvfp4_debug_gemm_skip_load(enable=True):
    """Failure-detection test hook (see include/nvfp4.h)."""
    lib().nvfp4_debug_gemm_skip_load(1 if enable else 0)


def nvfp4_debug_quantize_skip_load(pass_=2):
    """Quantiser failure-detection test hook (see include/nvfp4.h): 1 = amax
    pass, 2 = encode pass, 0 = off."""
    lib().nvfp4_debug_quantize_skip_load(int(pass_))


MMA_RATE_KINDS = {0: "nvf4 pair 256x256x64", 1: "nvf4 single 128x256x64", 2: "bf16 pair 256x256x16",
                  3: "bf16 single 128x256x16"}


def nvfp4_debug_mma_rate(kind, iters=4096):
    """Isolated tensor-core instruction rate on the current device (see
    include/nvfp4.h): returns (TFLOP/s, cycles per instruction)."""
    tf, cyc = ctypes.c_double(), ctypes.c_double()
    _check(lib().nvfp4_debug_mma_rate(int(kind), int(iters), ctypes.byref(tf), ctypes.byref(cyc)),
           "nvfp4_debug_mma_rate")
    return tf.value, cyc.value


def nvfp4_check_device_status(workspace, stream=None):
    """Synchronise, read and clear the workspace's device status word."""
    return lib().nvfp4_check_device_status(_ptr(workspace), _stream(stream))


# --- quantised AdamW state codec -------------------------------------------
@dataclass
class QAdamWState:
    """An optimizer moment stored in NVFP4 (see include/nvfp4.h)."""
    codes: torch.Tensor         # uint8 [rows, cols/2]
    sf: torch.Tensor            # uint8 [rows, cols/16] row-major
    tensor_scale: torch.Tensor  # float32 [1]
    tile_mean: torch.Tensor     # uint16 BF16 bits [rows/16, cols/16] (second moment), else empty
    rows: int
    cols: int


def _qadamw_empty(rows, cols, device, second):
    return QAdamWState(codes=torch.empty((rows, cols // 2), dtype=torch.uint8, device=device),
                       sf=torch.empty((rows, cols // 16), dtype=torch.uint8, device=device),
                       tensor_scale=torch.empty(1, dtype=torch.float32, device=device),
                       tile_mean=torch.empty((rows // 16, cols // 16) if second else (0,), dtype=torch.int16,
                                             device=device),
                       rows=rows, cols=cols)


def nvfp4_qadamw_workspace_size():
    n = ctypes.c_size_t(0)
    _check(lib().nvfp4_qadamw_workspace_size(ctypes.byref(n)), "nvfp4_qadamw_workspace_size")
    return n.value


def nvfp4_qadamw_m_encode(m, rht_seed, sr_seed, sr_offset=0, out=None, workspace=None, stream=None):
    """First moment m (float32 CUDA [rows, cols]) -> QAdamWState."""
    assert m.dtype == torch.float32 and m.dim() == 2 and m.is_contiguous()
    rows, cols = m.shape
    if out is None:
        out = _qadamw_empty(rows, cols, m.device, False)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_qadamw_workspace_size(), m.device)
    st = lib().nvfp4_qadamw_m_encode(_ptr(m), rows, cols, rht_seed, sr_seed, sr_offset, _ptr(out.codes),
                                     _ptr(out.sf), _ptr(out.tensor_scale), _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    _check(st, "nvfp4_qadamw_m_encode")
    return out


def nvfp4_qadamw_m_decode(state, rht_seed, out=None, stream=None):
    if out is None:
        out = torch.empty((state.rows, state.cols), dtype=torch.float32, device=state.codes.device)
    st = lib().nvfp4_qadamw_m_decode(_ptr(state.codes), _ptr(state.sf), _ptr(state.tensor_scale), state.rows,
                                     state.cols, rht_seed, _ptr(out), _stream(stream))
    _check(st, "nvfp4_qadamw_m_decode")
    return out


def nvfp4_qadamw_v_encode(v, rht_seed, out=None, workspace=None, stream=None):
    """Second moment v (float32 CUDA [rows, cols], >= 0) -> QAdamWState."""
    assert v.dtype == torch.float32 and v.dim() == 2 and v.is_contiguous()
    rows, cols = v.shape
    if out is None:
        out = _qadamw_empty(rows, cols, v.device, True)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_qadamw_workspace_size(), v.device)
    st = lib().nvfp4_qadamw_v_encode(_ptr(v), rows, cols, rht_seed, _ptr(out.codes), _ptr(out.sf),
                                     _ptr(out.tensor_scale), _ptr(out.tile_mean), _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    _check(st, "nvfp4_qadamw_v_encode")
    return out


def nvfp4_qadamw_v_decode(state, rht_seed, out=None, stream=None):
    if out is None:
        out = torch.empty((state.rows, state.cols), dtype=torch.float32, device=state.codes.device)
    st = lib().nvfp4_qadamw_v_decode(_ptr(state.codes), _ptr(state.sf), _ptr(state.tensor_scale),
                                     _ptr(state.tile_mean), state.rows, state.cols, rht_seed, _ptr(out),
                                     _stream(stream))
    _check(st, "nvfp4_qadamw_v_decode")
    return out


# --- LoRA-SVD projection -----------------------------------------------------
def nvfp4_lora_workspace_size(tokens, rank):
    n = ctypes.c_size_t(0)
    _check(lib().nvfp4_lora_workspace_size(tokens, rank, ctypes.byref(n)), "nvfp4_lora_workspace_size")
    return n.value


def nvfp4_lora_forward(xq, wq, x, l1, l2, beta, out_dtype=NVFP4_OUT_BF16, y=None, u=None, workspace=None,
                       stream=None):
    """Y = Q(X) Q(W_res)^T + beta BF16(X L1^T) L2^T (see include/nvfp4.h).
    x: BF16 [T, din] (unit column stride), l1 BF16 [r, din], l2 BF16 [dout, r]
    (contiguous).  Returns (y, u)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert l1.dtype == torch.bfloat16 and l1.is_contiguous() and l2.dtype == torch.bfloat16 and l2.is_contiguous()
    T, din = x.shape
    r = l1.shape[0]
    dout = wq.rows
    dev = x.device
    if y is None:
        dt = torch.float32 if out_dtype == NVFP4_OUT_F32 else torch.bfloat16
        y = torch.empty((T, dout), dtype=dt, device=dev)
    if u is None:
        u = torch.empty((T, r), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_lora_workspace_size(T, r), dev)
    ta, tb = xq._c(), wq._c()
    ldx = x.stride(0) if T > 1 else din
    ldy = y.stride(0) if T > 1 else dout
    st = lib().nvfp4_lora_forward(ctypes.byref(ta), ctypes.byref(tb), _ptr(x), ldx, _ptr(l1), _ptr(l2), r,
                                  float(beta), out_dtype, _ptr(y), ldy, _ptr(u), _ptr(workspace), workspace.numel(),
                                  _stream(stream))
    _check(st, "nvfp4_lora_forward")
    return y, u


# --- Newton-Schulz step (Q-Root) ---------------------------------------------
def nvfp4_abs_percentile_bf16(x, p=99.0, q=None, workspace=None, stream=None):
    """q[0] = nearest-rank p-th percentile of |x| (x: BF16 CUDA tensor, any
    shape, contiguous).  Returns q (float32 CUDA tensor [1])."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    if q is None:
        q = torch.empty(1, dtype=torch.float32, device=x.device)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check(lib().nvfp4_abs_percentile_workspace_size(ctypes.byref(n)), "nvfp4_abs_percentile_workspace_size")
        workspace = _alloc_ws(n.value, x.device)
    st = lib().nvfp4_abs_percentile_bf16(_ptr(x), x.numel(), float(p), _ptr(q), _ptr(workspace), workspace.numel(),
                                         _stream(stream))
    _check(st, "nvfp4_abs_percentile_bf16")
    return q


def nvfp4_clip_bf16(x, q, out=None, stream=None):
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    if out is None:
        out = torch.empty_like(x)
    _check(lib().nvfp4_clip_bf16(_ptr(x), x.numel(), _ptr(q), _ptr(out), _stream(stream)), "nvfp4_clip_bf16")
    return out


def nvfp4_axpby_bf16(x, y, a, b, out=None, stream=None):
    assert x.dtype == torch.bfloat16 and y.dtype == torch.bfloat16 and x.is_contiguous() and y.is_contiguous()
    assert x.numel() == y.numel()
    if out is None:
        out = torch.empty_like(x)
    _check(lib().nvfp4_axpby_bf16(_ptr(x), _ptr(y), x.numel(), float(a), float(b), _ptr(out), _stream(stream)),
           "nvfp4_axpby_bf16")
    return out


def nvfp4_ns_workspace_size(m, n):
    s = ctypes.c_size_t(0)
    _check(lib().nvfp4_ns_workspace_size(m, n, ctypes.byref(s)), "nvfp4_ns_workspace_size")
    return s.value


def nvfp4_ns_step(x, a, b, c, p=99.0, out=None, workspace=None, stream=None):
    """One Newton-Schulz step with NVFP4 products on the BF16 iterate x
    [m, n] (see include/nvfp4.h).  Returns X'."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    m, n = x.shape
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = _alloc_ws(nvfp4_ns_workspace_size(m, n), x.device)
    st = lib().nvfp4_ns_step(_ptr(x), m, n, float(a), float(b), float(c), float(p), _ptr(out), _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(st, "nvfp4_ns_step")
    return out
