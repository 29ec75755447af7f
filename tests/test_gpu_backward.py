"""bsq_linear_backward: both gradients of a linear layer from one grad_out, with output masks
(AstrAI `astrai/extension/fp8.py`, `_LinearFp8.backward`: dX and dW come from one gradient
and `needs_input_grad` decides which products run), on the dequantize-then-BF16-matmul
backward of MSLK PR #393, Implementation Method.

Each wanted product is checked against the float64 oracle with the parity tests' bound and
bit for bit against the single-product entry point (the fused launch runs the same tiles in
the same order); an output the mask leaves out is not touched (it keeps its NaN fill).
"""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_BF16, synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR]
X_, W_ = bsq.BSQ_NEEDS_GRAD_X, bsq.BSQ_NEEDS_GRAD_W


def _bits(t):
    return t.view(torch.int16)


def _run(G, W, X, needs, M, N, K):
    gx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    gw = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.linear_backward(G, W, X, needs, grad_x=gx, grad_w=gw)
    torch.cuda.synchronize()
    return gx, gw


@pytest.mark.parametrize("needs", [X_, W_, X_ | W_])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(300, 200, 352), (513, 136, 416), (64, 128, 256), (1100, 264, 640)])
def test_linear_backward_masks(fmt, M, N, K, needs):
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=80 + fmt, device="cpu")
    X = synth.make_packed(fmt, 1, M, K, 1.0, seed=81 + fmt, device="cpu")
    G = synth.randn((M, N), 1.0, 82, "cpu", torch.bfloat16)
    Gd, Wd, Xd = G.cuda(), W.to("cuda"), X.to("cuda")
    gx, gw = _run(Gd, Wd, Xd, needs, M, N, K)
    g = bf16_vals(G)
    if needs & X_:
        w = oracle_deq(W)[0]
        assert_gemm(bf16_vals(gx), Gm.dgrad(g, w), g, w, N, f"backward dgrad fmt={fmt}")
        assert torch.equal(_bits(gx), _bits(bsq.linear_dgrad(Gd, Wd)))
    else:
        assert torch.isnan(gx.float()).all(), "grad_x written although not asked for"
    if needs & W_:
        x = oracle_deq(X)[0]
        assert_gemm(bf16_vals(gw), Gm.wgrad(g, x), g, x, M, f"backward wgrad fmt={fmt}")
        assert torch.equal(_bits(gw), _bits(bsq.linear_wgrad(Gd, Xd)))
    else:
        assert torch.isnan(gw.float()).all(), "grad_w written although not asked for"
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


def test_linear_backward_mixed_formats_and_small_m():
    """Formats that differ (the FP8 tiny workload: W E4M3, X BF16) and M <= 16 take the two
    single-product kernels one after the other."""
    for fw, fx, M in [(synth.FMT_FP8, synth.FMT_BF16, 64), (synth.FMT_MXFP4, synth.FMT_MXFP4, 16),
                      (synth.FMT_NVFP4, synth.FMT_FP8, 5), (synth.FMT_FP8_TENSOR, synth.FMT_MXFP4, 40)]:
        N, K = 256, 512
        W = synth.make_packed(fw, 1, N, K, 0.5, seed=90, device="cpu")
        X = synth.make_packed(fx, 1, M, K, 1.0, seed=91, device="cpu")
        G = synth.randn((M, N), 1.0, 92, "cpu", torch.bfloat16)
        gx, gw = _run(G.cuda(), W.to("cuda"), X.to("cuda"), X_ | W_, M, N, K)
        g, w, x = bf16_vals(G), oracle_deq(W)[0], oracle_deq(X)[0]
        assert_gemm(bf16_vals(gx), Gm.dgrad(g, w), g, w, N, f"dgrad {fw}/{fx} M={M}")
        assert_gemm(bf16_vals(gw), Gm.wgrad(g, x), g, x, M, f"wgrad {fw}/{fx} M={M}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


def test_linear_backward_degenerate_sizes():
    K = 256
    W = synth.make_packed(synth.FMT_MXFP4, 1, 128, K, 1.0, seed=93, device="cpu").to("cuda")
    X = synth.make_packed(synth.FMT_MXFP4, 1, 0, K, 1.0, seed=94, device="cpu").to("cuda")
    G = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    gx, gw = _run(G, W, X, X_ | W_, 0, 128, K)
    assert (gw.float() == 0).all().item(), "M = 0: grad_w must be zeros"
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


def test_linear_backward_fp8_block_and_tensor_scales_share_a_launch():
    """W with 128 x 128 scale blocks and X with one scale per tensor run the same FP8
    kernels, so both products share one launch; each keeps its own scale layout."""
    M, N, K = 300, 264, 384
    W = synth.make_packed(synth.FMT_FP8, 1, N, K, 0.5, seed=95, device="cpu")
    X = synth.make_packed(synth.FMT_FP8_TENSOR, 1, M, K, 1.0, seed=96, device="cpu")
    G = synth.randn((M, N), 1.0, 97, "cpu", torch.bfloat16)
    Gd, Wd, Xd = G.cuda(), W.to("cuda"), X.to("cuda")
    gx, gw = _run(Gd, Wd, Xd, X_ | W_, M, N, K)
    g, w, x = bf16_vals(G), oracle_deq(W)[0], oracle_deq(X)[0]
    assert_gemm(bf16_vals(gx), Gm.dgrad(g, w), g, w, N, "dgrad (block scales)")
    assert_gemm(bf16_vals(gw), Gm.wgrad(g, x), g, x, M, "wgrad (per-tensor scale)")
    assert torch.equal(_bits(gx), _bits(bsq.linear_dgrad(Gd, Wd)))
    assert torch.equal(_bits(gw), _bits(bsq.linear_wgrad(Gd, Xd)))
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)
