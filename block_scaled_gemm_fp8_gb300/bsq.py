"""ctypes binding of libbsq.so (declared in include/bsq.h): same entry-point names, argument
marshalling only.  Every computation runs in the library's CUDA kernels; there is no
fallback path -- if the library or a GPU is missing, the calls raise.

Tensors are torch tensors on the current CUDA device; a packed operand is any object
with the attributes ``fmt, data, scale, tensor_scale, batch, rows, cols`` (for example
``block_scaled_gemm_fp8_gb300.synth.Packed``).
"""

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbsq.so")
HEADER_PATH = os.path.join(HERE, "..", "include", "bsq.h")

BSQ_BF16, BSQ_FP8_E4M3_B128, BSQ_MXFP4, BSQ_NVFP4, BSQ_FP8_E4M3_TENSOR, BSQ_FP8_E5M2_TENSOR = 0, 1, 2, 3, 4, 5
BSQ_OK, BSQ_ERR_INVALID_ARG, BSQ_ERR_UNSUPPORTED, BSQ_ERR_CUDA, BSQ_ERR_TIMEOUT = 0, 1, 2, 3, 4
BSQ_NEEDS_GRAD_X, BSQ_NEEDS_GRAD_W = 1, 2

_c_void_p, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32

SIGNATURES = {
    "bsq_dequant": [_i32, _c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p],
    "bsq_linear_dgrad": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p],
    "bsq_linear_wgrad": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p],
    "bsq_grouped_dgrad": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i64, _i64, _c_void_p,
                          _c_void_p, _c_void_p],
    "bsq_grouped_wgrad": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _i64,
                          _c_void_p, _c_void_p],
    "bsq_linear_backward": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p,
                            _c_void_p, _c_void_p, _i64, ctypes.c_uint32, _c_void_p, _c_void_p, _c_void_p],
    "bsq_linear_forward": [_i32, _c_void_p, _c_void_p, _c_void_p, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i64,
                           _i64, _c_void_p, _c_void_p],
    "bsq_linear_dgrad_smallm_noalloc": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i64,
                                        _c_void_p, _c_void_p],
    "bsq_quantize_e5m2": [_c_void_p, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p],
    "bsq_linear_backward_e5m2": [_c_void_p, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p,
                                 _c_void_p, _c_void_p, _i64, ctypes.c_uint32, _i32, _c_void_p, _c_void_p,
                                 _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p],
    "bsq_status_string": [_i32],
    "bsq_last_error": [],
    "bsq_get_device_error": [ctypes.POINTER(_i32), _c_void_p],
    "bsq_num_sms": [],
}
_RESTYPES = {"bsq_status_string": ctypes.c_char_p, "bsq_last_error": ctypes.c_char_p}


class BsqError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


_lib = None


def lib():
    """Load libbsq.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m block_scaled_gemm_fp8_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, _i32)
        _lib = L
    return _lib


def header_entry_points():
    """Names of the functions include/bsq.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsq_[a-z_]+)\s*\(", text)))


def status_string(s):
    return lib().bsq_status_string(int(s)).decode()


def last_error():
    return lib().bsq_last_error().decode()


def _check(status):
    if status != BSQ_OK:
        raise BsqError(status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def num_sms():
    return int(lib().bsq_num_sms())


def get_device_error(stream=None):
    """(status, code): synchronizes the stream and reads/clears the device error word."""
    code = _i32(0)
    st = lib().bsq_get_device_error(ctypes.byref(code), _stream(stream))
    return st, code.value


def dequant(p, out=None, stream=None):
    """BF16 [batch, rows, cols] from a packed operand."""
    if out is None:
        out = torch.empty((p.batch, p.rows, p.cols), dtype=torch.bfloat16, device=p.data.device)
    _check(lib().bsq_dequant(p.fmt, _ptr(p.data), _ptr(p.scale), _ptr(p.tensor_scale), p.batch, p.rows, p.cols,
                             _ptr(out), _stream(stream)))
    return out


def linear_dgrad(grad_out, w, out=None, stream=None):
    """grad_x[M,K] = grad_out[M,N] @ deq(W)[N,K]."""
    M, N = grad_out.shape
    if out is None:
        out = torch.empty((M, w.cols), dtype=torch.bfloat16, device=grad_out.device)
    _check(lib().bsq_linear_dgrad(_ptr(grad_out), M, N, w.fmt, _ptr(w.data), _ptr(w.scale), _ptr(w.tensor_scale),
                                  w.cols, _ptr(out), _stream(stream)))
    return out


def linear_dgrad_smallm_noalloc(grad_out, w, out=None, stream=None):
    """grad_x[M,K] = grad_out[M,N] @ deq(W)[N,K] for M <= 16 without any device allocation
    (split-K scratch in a static device array of the library; K <= 16384)."""
    M, N = grad_out.shape
    if out is None:
        out = torch.empty((M, w.cols), dtype=torch.bfloat16, device=grad_out.device)
    _check(lib().bsq_linear_dgrad_smallm_noalloc(_ptr(grad_out), M, N, w.fmt, _ptr(w.data), _ptr(w.scale),
                                                 _ptr(w.tensor_scale), w.cols, _ptr(out), _stream(stream)))
    return out


def linear_wgrad(grad_out, x, out=None, stream=None):
    """grad_w[N,K] = grad_out[M,N]^T @ deq(X)[M,K]."""
    M, N = grad_out.shape
    if out is None:
        out = torch.empty((N, x.cols), dtype=torch.bfloat16, device=grad_out.device)
    _check(lib().bsq_linear_wgrad(_ptr(grad_out), M, N, x.fmt, _ptr(x.data), _ptr(x.scale), _ptr(x.tensor_scale),
                                  x.cols, _ptr(out), _stream(stream)))
    return out


def linear_backward(grad_out, w, x, needs=BSQ_NEEDS_GRAD_X | BSQ_NEEDS_GRAD_W, grad_x=None, grad_w=None,
                    stream=None):
    """(grad_x, grad_w): grad_out @ deq(W) and grad_out^T @ deq(X), each only when `needs` asks
    for it (None otherwise); one launch when both are wanted and W and X share a format."""
    M, N = grad_out.shape
    K = (w if w is not None else x).cols
    if needs & BSQ_NEEDS_GRAD_X and grad_x is None:
        grad_x = torch.empty((M, K), dtype=torch.bfloat16, device=grad_out.device)
    if needs & BSQ_NEEDS_GRAD_W and grad_w is None:
        grad_w = torch.empty((N, K), dtype=torch.bfloat16, device=grad_out.device)
    f = lambda p, a: None if p is None else getattr(p, a)
    _check(lib().bsq_linear_backward(
        _ptr(grad_out), M, N, f(w, "fmt") or 0, _ptr(f(w, "data")), _ptr(f(w, "scale")), _ptr(f(w, "tensor_scale")),
        f(x, "fmt") or 0, _ptr(f(x, "data")), _ptr(f(x, "scale")), _ptr(f(x, "tensor_scale")), K, needs,
        _ptr(grad_x) if needs & BSQ_NEEDS_GRAD_X else None, _ptr(grad_w) if needs & BSQ_NEEDS_GRAD_W else None,
        _stream(stream)))
    return (grad_x if needs & BSQ_NEEDS_GRAD_X else None), (grad_w if needs & BSQ_NEEDS_GRAD_W else None)


def quantize_e5m2(g, margin=0, codes=None, deq=None, want_deq=True, stream=None):
    """Per-tensor E5M2 quantization of a BF16 gradient with its current amax:
    (codes u8, step f32[1], amax f32[1], deq bf16 or None), all on g's device."""
    dev = g.device
    if codes is None:
        codes = torch.empty(g.shape, dtype=torch.uint8, device=dev)
    if deq is None and want_deq:
        deq = torch.empty(g.shape, dtype=torch.bfloat16, device=dev)
    step = torch.empty(1, dtype=torch.float32, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    _check(lib().bsq_quantize_e5m2(_ptr(g), g.numel(), margin, _ptr(codes), _ptr(deq), _ptr(step), _ptr(amax),
                                   _stream(stream)))
    return codes, step, amax, deq


def linear_backward_e5m2(grad_out, w, x, needs=BSQ_NEEDS_GRAD_X | BSQ_NEEDS_GRAD_W, margin=0, grad_x=None,
                         grad_w=None, stream=None):
    """(grad_x, grad_w, step, amax): the backward on grad_out quantized once to E5M2 (step and
    amax are the quantization's, f32[1] on the device)."""
    M, N = grad_out.shape
    K = (w if w is not None else x).cols
    dev = grad_out.device
    if needs & BSQ_NEEDS_GRAD_X and grad_x is None:
        grad_x = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if needs & BSQ_NEEDS_GRAD_W and grad_w is None:
        grad_w = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    codes = torch.empty((M, N), dtype=torch.uint8, device=dev)
    deq = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    step = torch.empty(1, dtype=torch.float32, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    f = lambda p, a: None if p is None else getattr(p, a)
    _check(lib().bsq_linear_backward_e5m2(
        _ptr(grad_out), M, N, f(w, "fmt") or 0, _ptr(f(w, "data")), _ptr(f(w, "scale")), _ptr(f(w, "tensor_scale")),
        f(x, "fmt") or 0, _ptr(f(x, "data")), _ptr(f(x, "scale")), _ptr(f(x, "tensor_scale")), K, needs, margin,
        _ptr(codes), _ptr(deq), _ptr(step), _ptr(amax),
        _ptr(grad_x) if needs & BSQ_NEEDS_GRAD_X else None, _ptr(grad_w) if needs & BSQ_NEEDS_GRAD_W else None,
        _stream(stream)))
    return (grad_x if needs & BSQ_NEEDS_GRAD_X else None), (grad_w if needs & BSQ_NEEDS_GRAD_W else None), step, amax


def linear_forward(x, w, out=None, stream=None):
    """y[M,N] = deq(X)[M,K] @ deq(W)[N,K]^T; W packed, X packed of W's kind or BF16 (fmt 0)."""
    if out is None:
        out = torch.empty((x.rows, w.rows), dtype=torch.bfloat16, device=x.data.device)
    _check(lib().bsq_linear_forward(x.fmt, _ptr(x.data), _ptr(x.scale), _ptr(x.tensor_scale), x.rows, w.fmt,
                                    _ptr(w.data), _ptr(w.scale), _ptr(w.tensor_scale), w.rows, x.cols, _ptr(out),
                                    _stream(stream)))
    return out


def grouped_dgrad(grad_out, w, offsets, out=None, stream=None):
    """Per expert e: grad_x[r0:r1] = grad_out[r0:r1] @ deq(W[e]); rows past offsets[-1] untouched."""
    S, N = grad_out.shape
    if out is None:
        out = torch.empty((S, w.cols), dtype=torch.bfloat16, device=grad_out.device)
    _check(lib().bsq_grouped_dgrad(_ptr(grad_out), S, N, w.fmt, _ptr(w.data), _ptr(w.scale), _ptr(w.tensor_scale),
                                   w.batch, w.cols, _ptr(offsets), _ptr(out), _stream(stream)))
    return out


def grouped_wgrad(grad_out, x, offsets, E, out=None, stream=None):
    """Per expert e: grad_w[e] = grad_out[r0:r1]^T @ deq(X)[r0:r1]; empty experts give zeros."""
    S, N = grad_out.shape
    if out is None:
        out = torch.empty((E, N, x.cols), dtype=torch.bfloat16, device=grad_out.device)
    _check(lib().bsq_grouped_wgrad(_ptr(grad_out), S, N, x.fmt, _ptr(x.data), _ptr(x.scale), _ptr(x.tensor_scale),
                                   x.cols, _ptr(offsets), E, _ptr(out), _stream(stream)))
    return out
