"""The five workloads at full size on the GPU, in the launch configuration bench.py times.

Every row of each output is checked on a seeded sample of output columns: the oracle
dequantizes only those columns of the packed operand and forms the float64 products,
so every expert-boundary row is covered.  Rows past offsets[E-1] (none here: all five
workloads route every token) and empty experts are checked exactly.
"""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import dequant as D
from oracle import gemm as Gm
from tests._util import ORACLE_FMT, assert_gemm, bf16_vals

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

NCOLS = 40


def _cols(K, seed):
    rng = np.random.default_rng(seed)
    c = rng.choice(K, size=NCOLS - 2, replace=False)
    return np.unique(np.concatenate([c, [0, K - 1]]))


def _deq_cols(p, cols, b=0):
    d, s, ts = p.numpy()
    return D.dequant_cols(ORACLE_FMT[p.fmt], d, s, ts, p.rows, p.cols, cols, b, p.batch)


@pytest.fixture(scope="module", params=[2, 3, 4, 5])
def cfg(request):
    c = synth.make_config(request.param, device="cuda")
    yield c
    del c
    torch.cuda.empty_cache()


def test_full_size_sampled(cfg):
    c = cfg
    K, N = c["K"], c["N"]
    cols = _cols(K, 123)
    g = bf16_vals(c["G"])
    if not c["grouped"]:
        gx = bsq.linear_dgrad(c["G"], c["W"])
        gw = bsq.linear_wgrad(c["G"], c["X"])
        torch.cuda.synchronize()
        w = _deq_cols(c["W"], cols)
        assert_gemm(bf16_vals(gx[:, cols]), g @ w, g, w, N, f"{c['name']} dgrad")
        x = _deq_cols(c["X"], cols)
        assert_gemm(bf16_vals(gw[:, cols]), g.T @ x, g, x, c["M"], f"{c['name']} wgrad")
        if "G_small" in c:
            gs = bf16_vals(c["G_small"])
            out = bsq.linear_dgrad(c["G_small"], c["W"])
            torch.cuda.synchronize()
            assert_gemm(bf16_vals(out[:, cols]), gs @ w, gs, w, N, "small-M dgrad")
    else:
        offs = c["offsets"]
        od = torch.from_numpy(offs).cuda()
        gx = bsq.grouped_dgrad(c["G"], c["W"], od)
        gw = bsq.grouped_wgrad(c["G"], c["X"], od, c["E"]) if c["X"] is not None else None
        torch.cuda.synchronize()
        gxs = bf16_vals(gx[:, cols])
        x = _deq_cols(c["X"], cols) if c["X"] is not None else None
        for e in range(c["E"]):
            r0, r1 = Gm.expert_rows(offs, e)
            if r1 == r0:
                if gw is not None:
                    assert (bf16_vals(gw[e][:, cols]) == 0).all()
                continue
            w = _deq_cols(c["W"], cols, e)
            assert_gemm(gxs[r0:r1], g[r0:r1] @ w, g[r0:r1], w, N, f"{c['name']} dgrad e={e}")
            if gw is not None:
                xe = x[r0:r1]
                assert_gemm(bf16_vals(gw[e][:, cols]), g[r0:r1].T @ xe, g[r0:r1], xe, r1 - r0,
                            f"{c['name']} wgrad e={e}")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0
