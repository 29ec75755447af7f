"""bsq_linear_forward, Y = deq(X) @ deq(W)^T with both operands packed (the forward product the
backward entry points differentiate: MSLK PR #393, Summary, mslk::f4f4bf16), against the
float64 oracle with the parity tests' bound (Kc = K), and bit for bit where one-hot rows
of X pick single columns of W.  Shapes span several pair tiles with ragged M, N and K."""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import formats as F
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq

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
