"""The five workloads at full size on the GPU, in the launch configuration bench.py times.

Every row of each output is checked on a seeded sample of output columns that holds
four columns of every 128-column block (each block is one m-tile of the GEMM kernel, so
a wrong block of any CTA is seen): the oracle dequantizes only those columns of the
packed operand and forms the float64 products, so every expert-boundary row is covered.
Rows past offsets[E-1] (none here: all five workloads route every token) and empty
experts are checked exactly.  The forward on the two dense workloads (packed X, and a BF16
X as in the FP8 linear layer, whose own forward is checked whole) and the E5M2 backward on
the MXFP4 4096^3 one are checked the same way.
"""

import pytest
import torch

import numpy as np

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import dequant as D
from oracle import gemm as Gm
from oracle import quantize as Q
from tests._util import (ORACLE_FMT, assert_gemm, bf16_vals, block_cols, check_config_sampled, deq_cols, oracle_deq,
                         run_config)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

PER_BLOCK = 4


def _cols(K, seed):
    return block_cols(K, PER_BLOCK, seed)


@pytest.fixture(scope="module", params=[2, 3, 4, 5])
def cfg(request):
    c = synth.make_config(request.param, device="cuda")
    yield c
    del c
    torch.cuda.empty_cache()


def test_full_size_sampled(cfg):
    c = cfg
    outs = run_config(c)
    check_config_sampled(c, outs, _cols(c["K"], 123))
    if "G_small" in c:
        out = bsq.linear_dgrad(c["G_small"], c["W"])
        torch.cuda.synchronize()
        check_config_sampled(c, {"small_m": out}, _cols(c["K"], 124))
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


@pytest.mark.parametrize("n", [2, 3])
def test_forward_full_size_sampled(n):
    """bsq_linear_forward Y = deq(X) @ deq(W)^T on the two dense workloads' packed X and W
    at full size: every row of Y on four columns of every 128-column block (the oracle
    dequantizes X whole and only the sampled rows of W)."""
    c = synth.make_config(n, device="cuda")
    y = bsq.linear_forward(c["X"], c["W"])
    torch.cuda.synchronize()
    cols = _cols(c["N"], 125)
    W = c["W"]
    d, sc, ts = W.numpy()
    w = D.dequant_rows(ORACLE_FMT[W.fmt], d, sc, ts, W.rows, W.cols, cols)
    x = oracle_deq(c["X"])[0]
    got = bf16_vals(y[:, torch.from_numpy(cols).cuda()])
    assert_gemm(got, Gm.forward(x, w), x, w, c["K"], f"{c['name']} forward")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


@pytest.mark.parametrize("n", [1, 2, 3])
def test_forward_bf16_activation_full_size(n):
    """bsq_linear_forward with a BF16 X and a packed W: the FP8 linear workload's own layer
    (its X is BF16) compared on every element, and the two dense workloads' weights against
    a seeded BF16 activation of their X's shape and law, every row on four columns of every
    128-column block."""
    c = synth.make_config(n, device="cuda")
    if n == 1:
        X = c["X"]
    else:
        X = synth.make_packed(synth.FMT_BF16, 1, c["X"].rows, c["K"], {2: 1.0, 3: 0.02}[n], 150 + n, "cuda")
    assert X.fmt == synth.FMT_BF16
    y = bsq.linear_forward(X, c["W"])
    torch.cuda.synchronize()
    W = c["W"]
    cols = np.arange(c["N"]) if n == 1 else _cols(c["N"], 126)
    d, sc, ts = W.numpy()
    w = D.dequant_rows(ORACLE_FMT[W.fmt], d, sc, ts, W.rows, W.cols, cols)
    x = oracle_deq(X)[0]
    got = bf16_vals(y[:, torch.from_numpy(cols).cuda()])
    assert_gemm(got, Gm.forward(x, w), x, w, c["K"], f"{c['name']} forward, BF16 X")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


def test_e5m2_backward_full_size_sampled():
    """bsq_linear_backward_e5m2 on the MXFP4 4096^3 workload: step and amax equal the
    oracle's quantization of the whole gradient; both products of the E5M2-quantized
    gradient on four columns of every 128-column block, every row."""
    c = synth.make_config(2, device="cuda")
    gx, gw, step, amax = bsq.linear_backward_e5m2(c["G"], c["W"], c["X"])
    torch.cuda.synchronize()
    codes, rstep, ramax = Q.quantize_e5m2(bf16_vals(c["G"]))
    assert float(step.item()) == rstep and float(amax.item()) == ramax
    gq = D.dequant_values(D.FMT_E5M2_TENSOR, codes.reshape(1, c["M"], c["N"]), np.array([rstep], dtype=np.float32),
                          None, 1, c["M"], c["N"])[0]
    cols = _cols(c["K"], 126)
    sel = torch.from_numpy(cols).cuda()
    w, x = deq_cols(c["W"], cols), deq_cols(c["X"], cols)
    assert_gemm(bf16_vals(gx[:, sel]), Gm.dgrad(gq, w), gq, w, c["N"], "e5m2 dgrad 4096^3")
    assert_gemm(bf16_vals(gw[:, sel]), Gm.wgrad(gq, x), gq, x, c["M"], "e5m2 wgrad 4096^3")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0
