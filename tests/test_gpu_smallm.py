"""Split-K small-M dgrad (M <= 16 token rows) against the oracle.

These shapes force one to many row splits per column slab (N from 8 to 8192 rows),
ragged row ranges, a ragged last slab and repeated calls that reuse (and must leave
zeroed) the FP32 workspace."""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(16, 4096, 384), (1, 4096, 4096), (7, 304, 4096), (16, 2000, 96 * 2),
                                   (3, 16, 64), (16, 8, 4096), (16, 128, 4096), (5, 8192, 1024)])
def test_small_m_dgrad(fmt, M, N, K):
    if fmt != synth.FMT_FP8 and K % 32:
        pytest.skip("FP4 needs K % 32")
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=M + N + K, device="cpu")
    G = synth.randn((M, N), 1.0, 7, "cpu", torch.bfloat16)
    wd, gd = W.to("cuda"), G.cuda()
    w, g = oracle_deq(W)[0], bf16_vals(G)
    ref = Gm.dgrad(g, w)
    for rep in range(3):   # the workspace must be left zeroed after every call
        out = bsq.linear_dgrad(gd, wd)
        torch.cuda.synchronize()
        assert_gemm(bf16_vals(out), ref, g, w, N, f"small-M fmt={fmt} rep={rep}")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


def test_small_m_then_larger_k_grows_workspace():
    for K in (256, 8192, 512):
        W = synth.make_packed(synth.FMT_MXFP4, 1, 1024, K, 1.0, seed=K, device="cpu")
        G = synth.randn((16, 1024), 1.0, 8, "cpu", torch.bfloat16)
        out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
        torch.cuda.synchronize()
        w, g = oracle_deq(W)[0], bf16_vals(G)
        assert_gemm(bf16_vals(out), Gm.dgrad(g, w), g, w, 1024, f"K={K}")


def test_small_m_one_hot_rows_exact():
    N, K = 2048, 512
    W = synth.make_packed(synth.FMT_NVFP4, 1, N, K, 0.02, seed=9, device="cpu")
    idx = [0, 5, 1023, 2047]
    G = torch.zeros((len(idx), N), dtype=torch.bfloat16)
    for r, i in enumerate(idx):
        G[r, i] = 1.0
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_vals(out), oracle_deq(W)[0][idx])
