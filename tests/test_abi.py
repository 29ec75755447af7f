"""The C ABI on the CPU: the library loads, exports every entry point include/bsq.h
declares, and its host-side validation rejects bad arguments before touching a GPU
(no compute call runs here)."""

import ctypes
import os

import pytest

from block_scaled_gemm_fp8_gb300 import bsq

FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced by host validation


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(bsq.LIB_PATH):
        from block_scaled_gemm_fp8_gb300 import build
        build.build()
    return bsq.lib()


def test_exports_every_declared_entry_point(L):
    names = bsq.header_entry_points()
    assert set(names) >= {"bsq_dequant", "bsq_linear_dgrad", "bsq_linear_wgrad", "bsq_grouped_dgrad",
                          "bsq_grouped_wgrad", "bsq_status_string", "bsq_get_device_error"}
    for n in names:
        assert hasattr(L, n), n
    assert set(names) <= set(bsq.SIGNATURES), "binding is missing a declared entry point"


def test_status_strings(L):
    assert bsq.status_string(0) == "BSQ_OK"
    assert bsq.status_string(1) == "BSQ_ERR_INVALID_ARG"
    assert bsq.status_string(4) == "BSQ_ERR_TIMEOUT"
    assert bsq.status_string(99) == "BSQ_ERR_UNKNOWN"


def _dgrad(L, g=FAKE, M=64, N=128, fmt=1, w=FAKE, s=FAKE, ts=None, K=256, out=FAKE):
    return L.bsq_linear_dgrad(g, M, N, fmt, w, s, ts, K, out, None)


def test_validation_rejects_bad_arguments(L):
    assert _dgrad(L, g=None) == bsq.BSQ_ERR_INVALID_ARG
    assert _dgrad(L, out=None) == bsq.BSQ_ERR_INVALID_ARG
    assert _dgrad(L, out=FAKE + 8) == bsq.BSQ_ERR_INVALID_ARG        # misaligned
    assert _dgrad(L, fmt=9) == bsq.BSQ_ERR_INVALID_ARG
    assert _dgrad(L, M=-1) == bsq.BSQ_ERR_INVALID_ARG
    assert _dgrad(L, N=12) == bsq.BSQ_ERR_UNSUPPORTED               # grad_out row pitch not 16 B
    assert _dgrad(L, fmt=2, K=48) == bsq.BSQ_ERR_INVALID_ARG         # MXFP4 needs K % 32
    assert _dgrad(L, fmt=3, K=48) == bsq.BSQ_ERR_UNSUPPORTED         # NVFP4 K % 32 for TMA pitch
    assert _dgrad(L, fmt=3, ts=None) == bsq.BSQ_ERR_INVALID_ARG      # NVFP4 needs a tensor scale
    assert _dgrad(L, fmt=1, s=None) == bsq.BSQ_ERR_INVALID_ARG
    assert "bsq_linear_dgrad" in bsq.last_error()
    assert L.bsq_dequant(0, FAKE, None, None, 1, 4, 32, FAKE, None) == bsq.BSQ_ERR_UNSUPPORTED
    assert L.bsq_dequant(2, FAKE, FAKE, None, 1, 4, 48, FAKE, None) == bsq.BSQ_ERR_INVALID_ARG
    assert L.bsq_grouped_dgrad(FAKE, 16, 128, 1, FAKE, FAKE, None, 0, 256, FAKE, FAKE, None) == \
        bsq.BSQ_ERR_INVALID_ARG                                      # E = 0
    assert L.bsq_grouped_dgrad(FAKE, 16, 128, 1, FAKE, FAKE, None, 2000, 256, FAKE, FAKE, None) == \
        bsq.BSQ_ERR_UNSUPPORTED                                      # E above the limit
    assert L.bsq_grouped_wgrad(FAKE, 16, 128, 1, FAKE, FAKE, None, 256, None, 4, FAKE, None) == \
        bsq.BSQ_ERR_INVALID_ARG                                      # null offsets
    code = ctypes.c_int32(0)
    assert L.bsq_get_device_error(None, None) == bsq.BSQ_ERR_INVALID_ARG


def test_empty_problems_return_ok_without_launch(L):
    # K == 0 or M == 0 (dgrad) is a no-op that must not touch the device
    assert _dgrad(L, M=0) == bsq.BSQ_OK
    assert _dgrad(L, K=0) == bsq.BSQ_OK
    assert L.bsq_dequant(1, FAKE, FAKE, None, 0, 4, 32, FAKE, None) == bsq.BSQ_OK


def test_linear_backward_validation(L):
    def bw(needs, w=FAKE, x=FAKE, gx=FAKE, gw=FAKE, wf=1, xf=1):
        return L.bsq_linear_backward(FAKE, 64, 128, wf, w, FAKE, None, xf, x, FAKE, None, 256, needs, gx, gw, None)
    assert bw(0, w=None, x=None, gx=None, gw=None) == bsq.BSQ_OK          # nothing wanted: nothing read
    assert bw(4) == bsq.BSQ_ERR_INVALID_ARG                               # unknown mask bit
    assert bw(bsq.BSQ_NEEDS_GRAD_X, w=None) == bsq.BSQ_ERR_INVALID_ARG    # W needed for grad_x
    assert bw(bsq.BSQ_NEEDS_GRAD_W, x=None) == bsq.BSQ_ERR_INVALID_ARG    # X needed for grad_w
    assert bw(3, gw=None) == bsq.BSQ_ERR_INVALID_ARG
    assert bw(3, xf=9) == bsq.BSQ_ERR_INVALID_ARG
    assert "bsq_linear" in bsq.last_error()


def test_fp8_per_tensor_format_validation(L):
    assert _dgrad(L, fmt=4, K=40) == bsq.BSQ_ERR_UNSUPPORTED            # FP8 row pitch: K % 16
    assert _dgrad(L, fmt=4, s=FAKE + 2) == bsq.BSQ_ERR_INVALID_ARG       # scale_inv must be 4-byte aligned
    assert _dgrad(L, fmt=6) == bsq.BSQ_ERR_INVALID_ARG                   # no such format
    assert _dgrad(L, fmt=5) == bsq.BSQ_ERR_UNSUPPORTED                   # E5M2: the gradient's format only
    assert L.bsq_dequant(4, FAKE, FAKE + 4, None, 0, 4, 32, FAKE, None) == bsq.BSQ_OK
    # the allocation-free small-M entry point serves 128 x 128 FP8 blocks only
    assert L.bsq_linear_dgrad_smallm_noalloc(FAKE, 4, 64, 4, FAKE, FAKE, None, 256, FAKE, None) == \
        bsq.BSQ_ERR_UNSUPPORTED


def test_linear_forward_validation(L):
    def fw(xf=2, wf=2, M=64, N=128, K=256, y=FAKE):
        return L.bsq_linear_forward(xf, FAKE, FAKE, FAKE, M, wf, FAKE, FAKE, FAKE, N, K, y, None)
    assert fw(wf=0) == bsq.BSQ_ERR_UNSUPPORTED          # the weight is packed
    assert fw(xf=0, wf=0) == bsq.BSQ_ERR_UNSUPPORTED
    assert fw(xf=0, K=100) == bsq.BSQ_ERR_UNSUPPORTED   # BF16 X row pitch: K % 8
    assert fw(xf=0, wf=3, K=48) == bsq.BSQ_ERR_UNSUPPORTED   # NVFP4 W: K % 32
    assert fw(xf=0, M=0) == bsq.BSQ_OK                  # BF16 X with a packed W: accepted
    assert fw(xf=2, wf=3) == bsq.BSQ_ERR_UNSUPPORTED    # MXFP4 x NVFP4: no common kernel
    assert fw(N=12) == bsq.BSQ_ERR_UNSUPPORTED          # Y row pitch
    assert fw(y=None) == bsq.BSQ_ERR_INVALID_ARG
    assert fw(M=0) == bsq.BSQ_OK and fw(N=0) == bsq.BSQ_OK


def test_e5m2_gradient_validation(L):
    def q(g=FAKE, n=64, margin=0, codes=FAKE, deq=None, step=FAKE + 64, amax=FAKE + 128):
        return L.bsq_quantize_e5m2(g, n, margin, codes, deq, step, amax, None)
    assert q(margin=-1) == bsq.BSQ_ERR_INVALID_ARG and q(margin=31) == bsq.BSQ_ERR_INVALID_ARG
    assert q(n=-1) == bsq.BSQ_ERR_INVALID_ARG
    assert q(g=FAKE + 8) == bsq.BSQ_ERR_INVALID_ARG          # g must be 16-byte aligned
    assert q(codes=FAKE + 4) == bsq.BSQ_ERR_INVALID_ARG      # codes 8-byte aligned
    assert q(deq=FAKE + 8) == bsq.BSQ_ERR_INVALID_ARG        # deq 16-byte aligned
    assert q(step=None) == bsq.BSQ_ERR_INVALID_ARG and q(amax=FAKE + 2) == bsq.BSQ_ERR_INVALID_ARG
    # E5M2 is no GEMM operand and no forward operand
    assert L.bsq_linear_wgrad(FAKE, 64, 64, 5, FAKE, FAKE, None, 64, FAKE, None) == bsq.BSQ_ERR_UNSUPPORTED
    assert L.bsq_linear_forward(5, FAKE, FAKE, None, 64, 5, FAKE, FAKE, None, 64, 64, FAKE, None) == \
        bsq.BSQ_ERR_UNSUPPORTED
    # the E5M2 backward checks its products' operands before anything runs
    def bw(wf=2, xf=2, needs=3, deq=FAKE, N=64):
        return L.bsq_linear_backward_e5m2(FAKE, 64, N, wf, FAKE, FAKE, None, xf, FAKE, FAKE, None, 64, needs, 0,
                                          FAKE, deq, FAKE + 64, FAKE + 128, FAKE, FAKE, None)
    assert bw(needs=4) == bsq.BSQ_ERR_INVALID_ARG
    assert bw(deq=None) == bsq.BSQ_ERR_INVALID_ARG
    assert bw(wf=5) == bsq.BSQ_ERR_UNSUPPORTED and bw(xf=5, needs=2) == bsq.BSQ_ERR_UNSUPPORTED
    assert bw(N=12) == bsq.BSQ_ERR_UNSUPPORTED                # grad_out row pitch
    # dequantizing E5M2 codes: a per-tensor step, FP8 row pitch
    assert L.bsq_dequant(5, FAKE, FAKE + 4, None, 1, 4, 40, FAKE, None) == bsq.BSQ_ERR_UNSUPPORTED
    assert L.bsq_dequant(5, FAKE, FAKE + 2, None, 1, 4, 32, FAKE, None) == bsq.BSQ_ERR_INVALID_ARG
    assert L.bsq_dequant(5, FAKE, FAKE + 4, None, 0, 4, 32, FAKE, None) == bsq.BSQ_OK
