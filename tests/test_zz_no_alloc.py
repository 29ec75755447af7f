"""The allocation-free small-M dgrad entry point (bsq_linear_dgrad_smallm_noalloc).

It exists for callers that cannot call cudaMalloc (work recorded under stream capture,
hosts whose allocator owns all device memory).  Its split-K scratch is a static device
array of the library.  This test calls it through the C ABI twice in a row (the shared
scratch must be left clean by the first call) and checks each result against the
float64 oracle, grad_X = grad_out @ deq(W), within the tolerance the parity tests use,
and against the existing entry point bsq_linear_dgrad within that same tolerance.  The
file is named to be collected last and also passes when run alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import gemm as Gm
from tests._util import bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4])
@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (5, 1000, 512)])
def test_noalloc_matches_allocating_entry_point(fmt, M, N, K):
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=100 + M, device="cpu").to("cuda")
    G = synth.randn((M, N), 1.0, 101, "cuda", torch.bfloat16)
    existing = bsq.linear_dgrad(G, W)
    torch.cuda.synchronize()
    g = bf16_vals(G)
    w = oracle_deq(W.to("cpu"))[0]
    oracle = Gm.dgrad(g, w)
    # the parity tests' elementwise bound for this product: 2e-2 sqrt(N) rms(G) rms(W) plus
    # the output's BF16 rounding, and a relative Frobenius error of at most 5e-3
    bound = Gm.tolerance(N, g, w)
    lib = bsq.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.bsq_linear_dgrad_smallm_noalloc(_ptr(G), M, N, W.fmt, _ptr(W.data), _ptr(W.scale),
                                                 _ptr(W.tensor_scale), K, _ptr(out), stream)
        assert st == bsq.BSQ_OK, bsq.last_error()
        torch.cuda.synchronize()
        got = bf16_vals(out)
        ok, err, rel = Gm.check(got, oracle, bound)
        assert ok, f"call {call} vs oracle: max|err|={err} bound={bound} relF={rel}"
        ok, err, rel = Gm.check(got, bf16_vals(existing), bound)
        assert ok, f"call {call} vs bsq_linear_dgrad: max|err|={err} bound={bound} relF={rel}"
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = bsq.lib()
    W = synth.make_packed(synth.FMT_MXFP4, 1, 64, 16384 + 512, 1.0, seed=1, device="cpu").to("cuda")
    G = synth.randn((4, 64), 1.0, 2, "cuda", torch.bfloat16)
    out = torch.empty((4, W.cols), dtype=torch.bfloat16, device="cuda")
    st = lib.bsq_linear_dgrad_smallm_noalloc(_ptr(G), 4, 64, W.fmt, _ptr(W.data), _ptr(W.scale), None, W.cols,
                                             _ptr(out), None)
    assert st == bsq.BSQ_ERR_UNSUPPORTED and "16384" in bsq.last_error()
    G17 = synth.randn((17, 64), 1.0, 3, "cuda", torch.bfloat16)
    out17 = torch.empty((17, W.cols), dtype=torch.bfloat16, device="cuda")
    st = lib.bsq_linear_dgrad_smallm_noalloc(_ptr(G17), 17, 64, W.fmt, _ptr(W.data), _ptr(W.scale), None,
                                             W.cols, _ptr(out17), None)
    assert st == bsq.BSQ_ERR_UNSUPPORTED
