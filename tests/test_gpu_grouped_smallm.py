"""Grouped dgrad for decode-sized experts against the oracle.

bsq_grouped_dgrad sends a decode-sized call (S at most BSQ_GROUPED_SMALL_ROWS, default
64) wholly to the split-K small-M kernel; above that the pair-tile GEMM computes every row,
except that with BSQ_GROUPED_TAIL_ROWS = T > 0 each expert's ragged last tile of at most T
rows goes to the small-M kernel.  Both read the same device offsets (transformers PR
#50031 `FP8GroupedMatmulFunction.backward`: per expert, grad_out rows times the
dequantized expert weight).  Covered here:

  * S within the bound, so only the small-M kernel runs: experts with 0, 1, 15, 16, 17,
    33 and 40 rows (one to three 16-token passes), empty first and last experts, rows
    past offsets[E-1] never written;
  * both kernels in one call (T = 64): short last tiles (small-M) next to long ones
    (GEMM), with a GEMM part in front of a short tail (300 rows = 256 + 44);
  * the bounds moved: GEMM only; every expert below 256 rows and every short tail to
    small-M (T = 255); a 255-row call wholly to small-M (13 passes for a 200-row expert);
  * the 64 FP8 expert weights [64, 2816, 2048] of the grouped workload under a
    decode-sized batch (128 and 256 routed rows, the same Zipf law), every column checked;
  * malformed offsets: reported, nothing written;
  * a wait that runs out (test hook): the orderly abort, then a correct next call.
"""

import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR]
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_grouped(fmt, counts, N, K, seed, extra_rows=5, w_std=0.5):
    offsets = synth.offsets_from_counts(counts)
    E = len(counts)
    S = int(offsets[-1]) + extra_rows
    W = synth.make_packed(fmt, E, N, K, w_std, seed=seed, device="cpu")
    G = synth.randn((S, N), 1.0, seed + 1, "cpu", torch.bfloat16)
    if offsets[-1] < S:
        G[int(offsets[-1]):] = float("nan")          # never reaches a written row
    out = torch.full((S, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G.cuda(), W.to("cuda"), torch.from_numpy(offsets).cuda(), out=out)
    torch.cuda.synchronize()
    return offsets, W, G, bf16_vals(out)


def _check(offsets, W, G, got, N, what):
    w = oracle_deq(W)
    g = bf16_vals(G)
    ref = Gm.grouped_dgrad(g, w, offsets)
    used = int(offsets[-1])
    assert np.isnan(got[used:]).all(), f"{what}: rows past offsets[E-1] were written"
    for e in range(len(offsets)):
        r0, r1 = Gm.expert_rows(offsets, e)
        if r1 > r0:
            assert_gemm(got[r0:r1], ref[r0:r1], g[r0:r1], w[e], N, f"{what} expert {e}")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0, (what, st, code)


DECODE_COUNTS = [
    [0, 1, 15, 16, 17, 0, 3],                 # S 52: one and two passes, empty first expert
    [40, 0, 0, 2, 1, 0],                      # S 43: three passes, empty last experts
    [33] + [1] * 20 + [0] * 11,               # S 53: 32 experts, three passes for the first
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ci", range(len(DECODE_COUNTS)))
@pytest.mark.parametrize("N,K", [(200, 352), (1000, 2048)])
def test_decode_sized_experts_small_m_only(fmt, ci, N, K):
    if fmt != synth.FMT_FP8 and K % 32:
        pytest.skip("FP4 needs K % 32")
    counts = DECODE_COUNTS[ci]
    offsets, W, G, got = _run_grouped(fmt, counts, N, K, seed=500 + 10 * ci + fmt)
    _check(offsets, W, G, got, N, f"fmt={fmt} counts={ci}")


MIXED_COUNTS = [
    [300, 0, 5, 130, 64, 65, 256, 1],         # tails 44, 5, 64, 1 to small-M; 130, 65 to the GEMM
    [0, 600, 17],                             # 600 = 512 + 88 (GEMM), 17 (small-M)
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ci", range(len(MIXED_COUNTS)))
def test_small_m_and_gemm_in_one_call(fmt, ci, monkeypatch):
    monkeypatch.setenv("BSQ_GROUPED_TAIL_ROWS", "64")
    counts = MIXED_COUNTS[ci]
    N, K = 264, 384
    offsets, W, G, got = _run_grouped(fmt, counts, N, K, seed=600 + 10 * ci + fmt)
    _check(offsets, W, G, got, N, f"mixed fmt={fmt} counts={ci}")


@pytest.mark.parametrize("small,tail,counts", [
    ("0", "0", [0, 3, 200, 17, 255, 256, 300]),       # the GEMM takes every row
    ("0", "255", [0, 3, 200, 17, 255, 256, 300]),     # every expert below 256 rows, and 300's tail, to small-M
    ("255", "0", [0, 3, 200, 17, 30]),                # S = 255: the whole call to small-M
])
@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_NVFP4])
def test_bounds_move_rows_between_kernels(fmt, small, tail, counts, monkeypatch):
    monkeypatch.setenv("BSQ_GROUPED_SMALL_ROWS", small)
    monkeypatch.setenv("BSQ_GROUPED_TAIL_ROWS", tail)
    N, K = 192, 256
    offsets, W, G, got = _run_grouped(fmt, counts, N, K, seed=700 + fmt)
    _check(offsets, W, G, got, N, f"small={small} tail={tail} fmt={fmt}")


@pytest.mark.parametrize("rows", [128, 256])
def test_grouped_workload_weights_decode_batch(rows):
    """The 64 FP8 expert weights [64, 2816, 2048] with a decode-sized batch routed by the
    grouped workload's Zipf(1.1) law; every output element against the oracle."""
    c = synth.make_config(4, device="cpu", rows=rows)
    G, W, offsets = c["G"], c["W"], c["offsets"]
    S, K, N = c["M"], c["K"], c["N"]
    out = torch.full((S, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G.cuda(), W.to("cuda"), torch.from_numpy(offsets).cuda(), out=out)
    torch.cuda.synchronize()
    got = bf16_vals(out)
    g = bf16_vals(G)
    for e in range(c["E"]):
        r0, r1 = Gm.expert_rows(offsets, e)
        if r1 == r0:
            continue
        w = oracle_deq(synth.Packed(W.fmt, W.data[e:e + 1], W.scale[e:e + 1], None, 1, N, K))[0]
        ref = Gm.dgrad(g[r0:r1], w)
        assert_gemm(got[r0:r1], ref, g[r0:r1], w, N, f"decode batch {rows}, expert {e}")
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0


def test_bad_offsets_reported_nothing_written(monkeypatch):
    N, K, S = 128, 256, 40
    W = synth.make_packed(synth.FMT_MXFP4, 3, N, K, 1.0, seed=80, device="cpu").to("cuda")
    G = synth.randn((S, N), 1.0, 81, "cpu", torch.bfloat16).cuda()
    out = torch.full((S, K), 7.0, dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G, W, torch.tensor([10, 5, 30], dtype=torch.int32, device="cuda"), out=out)
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_ERR_INVALID_ARG and code == 2
    assert (out.float() == 7.0).all()
    bsq.grouped_dgrad(G, W, torch.tensor([10, 20, 41], dtype=torch.int32, device="cuda"), out=out)
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_ERR_INVALID_ARG and code == 2
    assert (out.float() == 7.0).all()
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0
    # S above the bound with a tail bound set: the GEMM and the small-M kernel both run,
    # both see the bad offsets
    monkeypatch.setenv("BSQ_GROUPED_TAIL_ROWS", "64")
    S2 = 300
    G2 = synth.randn((S2, N), 1.0, 82, "cpu", torch.bfloat16).cuda()
    out2 = torch.full((S2, K), 7.0, dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G2, W, torch.tensor([10, 290, 280], dtype=torch.int32, device="cuda"), out=out2)
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_ERR_INVALID_ARG and code == 2
    assert (out2.float() == 7.0).all()


TIMEOUT_SCRIPT = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, {root!r})
    import torch
    from block_scaled_gemm_fp8_gb300 import bsq, synth
    from oracle import gemm as Gm
    from tests._util import assert_gemm, bf16_vals, oracle_deq

    W = synth.make_packed(synth.FMT_NVFP4, 3, 1024, 512, 0.5, seed=1, device="cpu")
    W1 = synth.make_packed(synth.FMT_NVFP4, 1, 1024, 512, 0.5, seed=2, device="cpu")
    G = synth.randn((40, 1024), 1.0, 3, "cpu", torch.bfloat16)
    offs = synth.offsets_from_counts([20, 0, 20])
    wd, w1d, gd, od = W.to("cuda"), W1.to("cuda"), G.cuda(), torch.from_numpy(offs).cuda()
    g8d = gd[:8].contiguous()
    g, w, w1 = bf16_vals(G), oracle_deq(W), oracle_deq(W1)[0]
    calls = {{
        "linear_dgrad_m8": lambda: bsq.linear_dgrad(g8d, w1d),
        "grouped_dgrad_decode": lambda: bsq.grouped_dgrad(gd, wd, od),
    }}
    for name, call in calls.items():
        os.environ["BSQ_WAIT_LIMIT_MS"] = "50"
        os.environ["BSQ_TEST_DROP_CHUNK"] = "1"
        call()
        st, code = bsq.get_device_error()
        assert st == bsq.BSQ_ERR_TIMEOUT and code == 1, (name, st, code)
        del os.environ["BSQ_WAIT_LIMIT_MS"], os.environ["BSQ_TEST_DROP_CHUNK"]
        out = call()
        torch.cuda.synchronize()
        got = bf16_vals(out)
        if name == "linear_dgrad_m8":
            assert_gemm(got, Gm.dgrad(g[:8], w1), g[:8], w1, 1024, name)
        else:
            ref = Gm.grouped_dgrad(g, w, offs)
            for e in (0, 2):
                r0, r1 = Gm.expert_rows(offs, e)
                assert_gemm(got[r0:r1], ref[r0:r1], g[r0:r1], w[e], 1024, name)
        st, code = bsq.get_device_error()
        assert st == bsq.BSQ_OK and code == 0, (name, "after recovery", st, code)
        print("ok", name)
""")


def test_small_m_wait_runs_out_then_next_call_is_correct():
    """BSQ_TEST_DROP_CHUNK=1 withholds every CTA's first chunk (a copy nothing issues), so
    its wait runs out after a 50 ms limit: the kernel records BSQ_DEVERR_TIMEOUT, lets its
    other copies land, meets its cluster at both barriers and writes nothing; the next
    call with the hook off is correct.  Child process, so the settings touch no other test."""
    env = {k: v for k, v in os.environ.items() if not k.startswith("BSQ_")}
    r = subprocess.run([sys.executable, "-c", TIMEOUT_SCRIPT.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 2, r.stdout
