"""Split-K small-M dgrad (M <= 16 token rows) against the oracle.

These shapes force one to eight row splits per column slab (N from 8 to 14336 rows, one
to 32 chunks of 64 rows per split, so the chunk ring both fills and wraps), ragged row
ranges, a ragged last slab, repeated calls, and calls on two streams at once (the splits
add up inside a thread-block cluster, with no state shared between calls)."""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR]


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


def test_small_m_successive_shapes():
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


def test_small_m_ffn_weight():
    """M = 16 against the NVFP4 FFN weight (N 14336, K 5120): 32 chunks per split, the
    ring wraps four times."""
    N, K = 14336, 5120
    W = synth.make_packed(synth.FMT_NVFP4, 1, N, K, 0.02, seed=17, device="cpu")
    G = synth.randn((16, N), 1e-2, 18, "cpu", torch.bfloat16)
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    w, g = oracle_deq(W)[0], bf16_vals(G)
    assert_gemm(bf16_vals(out), Gm.dgrad(g, w), g, w, N, "small-M FFN weight")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


def test_small_m_concurrent_streams():
    """Two small-M dgrads in flight at once on two streams (different weights and shapes):
    each matches the oracle."""
    cases = [(synth.FMT_MXFP4, 16, 4096, 4096, 21), (synth.FMT_FP8, 9, 3000, 2048, 22)]
    data = []
    for fmt, M, N, K, seed in cases:
        W = synth.make_packed(fmt, 1, N, K, 0.5, seed=seed, device="cpu")
        G = synth.randn((M, N), 1.0, seed + 1, "cpu", torch.bfloat16)
        data.append((W, G, W.to("cuda"), G.cuda()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for rep in range(4):
        for (W, G, wd, gd), s in zip(data, streams):
            with torch.cuda.stream(s):
                outs.append((rep, W, G, bsq.linear_dgrad(gd, wd, stream=s)))
    torch.cuda.synchronize()
    for rep, W, G, out in outs:
        w, g = oracle_deq(W)[0], bf16_vals(G)
        assert_gemm(bf16_vals(out), Gm.dgrad(g, w), g, w, W.rows, f"concurrent rep={rep} fmt={W.fmt}")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0
