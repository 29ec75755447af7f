"""Repeated full-size runs of the pair-MMA GEMM kernels: against the oracle and against
themselves.

The tensor-core work of the GEMM kernels runs on pairs of SMs, and one CTA's operands
are read by an MMA the other CTA issues.  A fault in the protocol that hands operands
from one CTA to the other shows as one CTA's 128 x 256 block of some tile being wrong in
some runs, not in every run.  So each workload here runs once and is checked against the
float64 oracle on four columns of every 128-column block (every m-tile of every CTA),
then runs REPS more times into buffers refilled with NaN; every tile's accumulation order
is fixed, so each repeat must equal the first run bit for bit over the whole output.

Workloads: MXFP4 4096^3 dense dgrad and wgrad, as one fused backward launch and as the two
single-product launches, and the 128-expert MXFP4 grouped dgrad and wgrad (Dirichlet(0.3)
routing, empty experts; its wgrad takes the short-tile kernel).

A second test repeats the grouped workloads while another stream copies 2 GB buffers, so
that the kernels' loads meet a busy memory system at varying moments.  A result that
depends on when a load completes relative to the refill of its buffer (a ring slot read
with plain loads and refilled by TMA without an order between the two) differs from the
clean run there.

A third test repeats the forward kernel (same pair protocol) with a packed X and with a
BF16 X, half of the repeats under the same concurrent copies.
"""

import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from tests._util import block_cols, check_config_sampled, run_config

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

REPS = 20


@pytest.fixture(scope="module", params=[2, 5])
def cfg(request):
    c = synth.make_config(request.param, device="cuda")
    yield c
    del c
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fused", [True, False])
def test_repeats_match_oracle_and_first_run(cfg, fused):
    c = cfg
    if c["grouped"] and not fused:
        pytest.skip("the grouped workload has one launch per product either way")
    first = run_config(c, fused=fused)
    check_config_sampled(c, first, block_cols(c["K"], 4, 7))
    ref = {k: v.clone() for k, v in first.items()}
    bad = []
    for rep in range(REPS):
        for v in first.values():
            v.fill_(float("nan"))
        run_config(c, first, fused=fused)
        for k, v in first.items():
            if not torch.equal(v.view(torch.int16), ref[k].view(torch.int16)):
                diff = (v.view(torch.int16) != ref[k].view(torch.int16))
                bad.append((rep, k, int(diff.sum().item())))
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0, (st, code)
    assert not bad, f"{c['name']}: repeats that differ from the first run (rep, op, elements): {bad}"


@pytest.mark.parametrize("n", [4, 5])
def test_repeats_under_concurrent_memory_traffic_match_first_run(n):
    c = synth.make_config(n, device="cuda")
    first = run_config(c)
    ref = {k: v.clone() for k, v in first.items()}
    src = torch.empty(1 << 31, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    side = torch.cuda.Stream()
    bad = []
    for rep in range(6):
        for v in first.values():
            v.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            for _ in range(1 + rep % 3):
                dst.copy_(src)
                src.copy_(dst)
        if rep % 2:
            torch.cuda._sleep(20000 * rep)   # vary where the copies overlap the launch
        run_config(c, first)
        for k, v in first.items():
            if not torch.equal(v.view(torch.int16), ref[k].view(torch.int16)):
                bad.append((rep, k, int((v.view(torch.int16) != ref[k].view(torch.int16)).sum().item())))
    torch.cuda.synchronize()
    del src, dst
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0, (st, code)
    assert not bad, f"{c['name']}: repeats under concurrent traffic that differ from the clean run: {bad}"


@pytest.mark.parametrize("x_bf16", [False, True])
def test_forward_repeats_match_oracle_and_first_run(x_bf16):
    """The forward kernel's pair protocol, repeated: Y = X W^T on the MXFP4 4096^3 workload's
    W with its packed X or a BF16 X (TMA into the A ring, its own producer warp), the first
    run against the oracle on four columns of every 128-column block, then REPS runs into
    NaN-filled buffers, every other one while another stream copies 2 GB buffers; each must
    equal the first bit for bit."""
    from oracle import dequant as D
    from oracle import gemm as Gm
    from tests._util import ORACLE_FMT, assert_gemm, bf16_vals, oracle_deq
    c = synth.make_config(2, device="cuda")
    X = synth.make_packed(synth.FMT_BF16, 1, c["M"], c["K"], 1.0, 160, "cuda") if x_bf16 else c["X"]
    y = bsq.linear_forward(X, c["W"])
    torch.cuda.synchronize()
    cols = block_cols(c["N"], 4, 161)
    W = c["W"]
    d, sc, ts = W.numpy()
    w = D.dequant_rows(ORACLE_FMT[W.fmt], d, sc, ts, W.rows, W.cols, cols)
    x = oracle_deq(X)[0]
    assert_gemm(bf16_vals(y[:, torch.from_numpy(cols).cuda()]), Gm.forward(x, w), x, w, c["K"],
                f"forward bf16_x={x_bf16}")
    ref = y.clone()
    src = torch.empty(1 << 31, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    side = torch.cuda.Stream()
    bad = []
    for rep in range(REPS):
        y.fill_(float("nan"))
        torch.cuda.synchronize()
        if rep % 2:
            with torch.cuda.stream(side):
                dst.copy_(src)
            torch.cuda._sleep(10000 * (rep % 5))
        bsq.linear_forward(X, c["W"], out=y)
        if not torch.equal(y.view(torch.int16), ref.view(torch.int16)):
            bad.append((rep, int((y.view(torch.int16) != ref.view(torch.int16)).sum().item())))
    torch.cuda.synchronize()
    del src, dst
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0, (st, code)
    assert not bad, f"forward bf16_x={x_bf16}: repeats that differ from the first run (rep, elements): {bad}"
