"""bsq_linear_forward, Y = deq(X) @ deq(W)^T with both operands packed (the forward product the
backward entry points differentiate: MSLK PR #393, Summary, mslk::f4f4bf16) or with a BF16
X and a packed W (the FP8 linear layer of transformers PR #50031, whose activation is
BF16), against the float64 oracle with the parity tests' bound (Kc = K), and bit for bit
where one-hot rows of X pick single columns of W (edge and NaN scales included).  Shapes
span several pair tiles with ragged M, N and K."""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import formats as F
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq
from tests.test_gpu_edge_scales import KINDS, PACKED, assert_bits, expected_one_hot

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(300, 200, 352), (1, 8, 64), (600, 520, 1024), (129, 264, 96), (256, 256, 4096)])
def test_linear_forward(fmt, M, N, K):
    if fmt in (synth.FMT_MXFP4, synth.FMT_NVFP4) and K % 32:
        pytest.skip("FP4 needs K % 32")
    X = synth.make_packed(fmt, 1, M, K, 1.0, seed=120 + fmt, device="cpu")
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=121 + fmt, device="cpu")
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.linear_forward(X.to("cuda"), W.to("cuda"), out=y)
    torch.cuda.synchronize()
    x, w = oracle_deq(X)[0], oracle_deq(W)[0]
    assert_gemm(bf16_vals(y), Gm.forward(x, w), x, w, K, f"forward fmt={fmt}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


def test_linear_forward_mixed_fp8_scales():
    M, N, K = 300, 136, 512
    X = synth.make_packed(synth.FMT_FP8_TENSOR, 1, M, K, 1.0, seed=130, device="cpu")
    W = synth.make_packed(synth.FMT_FP8, 1, N, K, 0.5, seed=131, device="cpu")
    y = bsq.linear_forward(X.to("cuda"), W.to("cuda"))
    torch.cuda.synchronize()
    x, w = oracle_deq(X)[0], oracle_deq(W)[0]
    assert_gemm(bf16_vals(y), Gm.forward(x, w), x, w, K, "forward FP8 per-tensor x block")


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4])
def test_linear_forward_one_hot_rows_are_weight_columns(fmt):
    """Row i of X holds one nonzero, x_i at column k_i, so Y[i, :] is the single product
    x_i * deq(W)[:, k_i] (exact in FP32), rounded once to BF16: compared bit for bit."""
    M, N, K = 40, 264, 256
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=132, device="cpu")
    xf = torch.zeros((1, M, K))
    ks = np.random.default_rng(5).integers(0, K, size=M)
    xf[0, torch.arange(M), torch.from_numpy(ks)] = 1.0
    X = synth.quantize(fmt, xf)
    y = bsq.linear_forward(X.to("cuda"), W.to("cuda"))
    torch.cuda.synchronize()
    x = oracle_deq(X)[0]
    xi = x[np.arange(M), ks]
    assert np.count_nonzero(x) == M and (xi != 0).all()
    w = oracle_deq(W)[0]
    np.testing.assert_array_equal(bf16_vals(y), F.bf16_round(xi[:, None] * w[:, ks].T))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(300, 200, 352), (1, 8, 64), (600, 520, 1024), (129, 264, 96), (256, 256, 4096)])
def test_linear_forward_bf16_activation(fmt, M, N, K):
    """X in BF16 (the activation of a layer whose weight alone is quantized, as in the FP8
    linear layer of transformers PR #50031): Y = X @ deq(W)^T, X through TMA, W decoded."""
    if fmt in (synth.FMT_MXFP4, synth.FMT_NVFP4) and K % 32:
        pytest.skip("FP4 needs K % 32")
    X = synth.make_packed(synth.FMT_BF16, 1, M, K, 1.0, seed=140 + fmt, device="cpu")
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=141 + fmt, device="cpu")
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.linear_forward(X.to("cuda"), W.to("cuda"), out=y)
    torch.cuda.synchronize()
    x, w = oracle_deq(X)[0], oracle_deq(W)[0]
    assert_gemm(bf16_vals(y), Gm.forward(x, w), x, w, K, f"forward bf16 X fmt={fmt}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


def _one_hot_x(M, K, seed):
    rng = np.random.default_rng(seed)
    ks = rng.integers(0, K, size=M)
    ks[:3] = [0, K - 1, K // 2]
    xf = torch.zeros((1, M, K))
    xf[0, torch.arange(M), torch.from_numpy(ks)] = 1.0
    return xf, ks


@pytest.mark.parametrize("x_bf16", [True, False])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
def test_linear_forward_one_hot_edge_scales(fmt, kind, x_bf16):
    """W from synth.random_codes with slow-path and NaN scales (the decode paths quantized
    N(0, s) weights never take), X one-hot along K (BF16, or packed in W's kind): each
    element of Y is one dequantized W element, compared on BF16 bits against the oracle
    (IEEE NaN / infinity rules for the zero products, as in test_gpu_edge_scales)."""
    M, N, K = 70, 264, 384      # ragged N (two n-tiles, the second partly outside W), 6 k-blocks
    W = synth.random_codes(fmt, 1, N, K, seed=370 + fmt, scale_kind=kind)
    xf, ks = _one_hot_x(M, K, 371)
    X = synth.quantize(synth.FMT_BF16 if x_bf16 else fmt, xf)
    assert (oracle_deq(X)[0][np.arange(M), ks] == 1.0).all()
    y = bsq.linear_forward(X.to("cuda"), W.to("cuda"))
    torch.cuda.synchronize()
    assert_bits(y, expected_one_hot(oracle_deq(W)[0].T, ks), f"forward fmt={fmt} {kind} bf16_x={x_bf16}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)
