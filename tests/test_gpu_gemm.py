"""Fused dequant + tensor-core GEMMs on the GPU against the float64 oracle.

Bound (from the method's acceptance rule): |err| <= 2e-2 * sqrt(Kc) * rms(A) * rms(B)
elementwise and ||err||_F / ||ref||_F <= 5e-3, with A, B the BF16 operands of the product
and Kc its contraction length; closed forms (one-hot rows, zero gradients, empty experts)
are checked exactly.  Sizes span several tiles (128 x 256 x 64) and ragged tails.
"""

import json
import os

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import gemm as Gm
from tests._util import assert_gemm, bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_BF16, synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR]
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def _no_device_error():
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0, (st, code)


def _grad(M, N, seed, std=1.0):
    return synth.randn((M, N), std, seed, "cpu", torch.bfloat16)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(300, 200, 352), (16, 512, 256), (1, 64, 128), (513, 136, 416)])
def test_linear_dgrad(fmt, M, N, K):
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=11 + fmt, device="cpu")
    G = _grad(M, N, 12)
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    w = oracle_deq(W)[0]
    g = bf16_vals(G)
    assert_gemm(bf16_vals(out), Gm.dgrad(g, w), g, w, N, f"dgrad fmt={fmt}")
    _no_device_error()


# wgrad of a packed format has two kernels (default and short-tile, opt-in); "auto" leaves
# BSQ_GEMM_SHORT_TILES unset, "0" / "1" set it.
KERNELS = ["auto", "0", "1"]


def _select_kernel(monkeypatch, kernel):
    if kernel == "auto":
        monkeypatch.delenv("BSQ_GEMM_SHORT_TILES", raising=False)
    else:
        monkeypatch.setenv("BSQ_GEMM_SHORT_TILES", kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(300, 200, 352), (100, 520, 256), (1, 64, 128), (64, 128, 256), (1100, 264, 640)])
def test_linear_wgrad(fmt, M, N, K, kernel, monkeypatch):
    _select_kernel(monkeypatch, kernel)
    X = synth.make_packed(fmt, 1, M, K, 1.0, seed=21 + fmt, device="cpu")
    G = _grad(M, N, 22)
    out = bsq.linear_wgrad(G.cuda(), X.to("cuda"))
    torch.cuda.synchronize()
    x = oracle_deq(X)[0]
    g = bf16_vals(G)
    assert_gemm(bf16_vals(out), Gm.wgrad(g, x), g, x, M, f"wgrad fmt={fmt}")
    _no_device_error()


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4])
def test_one_hot_rows_are_exact_weight_rows(fmt):
    N, K = 384, 256
    W = synth.make_packed(fmt, 1, N, K, 1.0, seed=5, device="cpu")
    idx = [0, 1, 127, 128, 255, 383]
    G = torch.zeros((len(idx), N), dtype=torch.bfloat16)
    for r, i in enumerate(idx):
        G[r, i] = 1.0
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_vals(out), oracle_deq(W)[0][idx])


def test_zero_gradient_gives_exact_zero():
    W = synth.make_packed(synth.FMT_NVFP4, 1, 256, 512, 1.0, seed=6, device="cpu")
    G = torch.zeros((77, 256), dtype=torch.bfloat16)
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    X = synth.make_packed(synth.FMT_NVFP4, 1, 77, 512, 1.0, seed=7, device="cpu")
    outw = bsq.linear_wgrad(G.cuda(), X.to("cuda"))
    torch.cuda.synchronize()
    assert (bf16_vals(out) == 0).all() and (bf16_vals(outw) == 0).all()


def test_fp8_linear_page_example_ones_gradient():
    """transformers PR #50031 test_linear_backward_goes_through_dequantized_weight:
    FP8Linear(256 -> 384), 128x128 blocks, grid rand(3,2)+0.5, x [1,5,256], sum().backward()."""
    ex = GOLDEN["fp8_linear_example"]
    N, K = ex["out_features"], ex["in_features"]
    g = torch.Generator().manual_seed(0)
    codes = torch.randn(N, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    grid = torch.rand(*ex["scale_grid"], generator=g) + 0.5
    W = synth.Packed(synth.FMT_FP8, codes.reshape(1, N, K).contiguous(), grid.reshape(1, 3, 2).contiguous(), None, 1, N, K)
    tokens = int(np.prod(ex["input_shape"][:-1]))
    G = torch.ones((tokens, N), dtype=torch.bfloat16)
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    w = oracle_deq(W)[0]
    ref = Gm.dgrad(np.ones((tokens, N)), w)
    assert_gemm(bf16_vals(out), ref, np.ones((tokens, N)), w, N, "page example")
    # the page's own check: fp32 dequantized weight, rtol 1e-2, atol 1e-1
    wf = codes.view(torch.float8_e4m3fn).float() * grid.repeat_interleave(128, 0).repeat_interleave(128, 1)
    torch.testing.assert_close(out.float().cpu(), torch.ones(tokens, N) @ wf, rtol=ex["tolerance"]["rtol"],
                               atol=ex["tolerance"]["atol"])


def _grouped_inputs(fmt, counts, S, N, K, seed, tail_nan=True):
    offsets = synth.offsets_from_counts(counts)
    E = len(counts)
    W = synth.make_packed(fmt, E, N, K, 0.5, seed=seed, device="cpu")
    G = _grad(S, N, seed + 1)
    if tail_nan and offsets[-1] < S:
        G[int(offsets[-1]):] = float("nan")
    return offsets, W, G


GROUPED_COUNTS = [
    [0, 5, 0, 127, 128, 129, 1, 0, 300, 2],      # empty first / middle / last-but-one, tile edges
    [0, 0, 0],                                   # all experts empty
    [700],                                       # one expert = linear
    [1] * 40 + [0] * 3 + [257],                  # many tiny experts
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ci", range(len(GROUPED_COUNTS)))
def test_grouped_dgrad(fmt, ci):
    counts = GROUPED_COUNTS[ci]
    S, N, K = sum(counts) + 9, 200, 352                      # 9 rows past offsets[E-1]
    offsets, W, G = _grouped_inputs(fmt, counts, S, N, K, seed=30 + ci)
    out = torch.full((S, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G.cuda(), W.to("cuda"), torch.from_numpy(offsets).cuda(), out=out)
    torch.cuda.synchronize()
    got = bf16_vals(out)
    w = oracle_deq(W)
    g = bf16_vals(G)
    ref = Gm.grouped_dgrad(g, w, offsets)
    used = int(offsets[-1])
    assert np.isnan(got[used:]).all(), "rows past offsets[E-1] were written"
    for e in range(len(counts)):
        r0, r1 = Gm.expert_rows(offsets, e)
        if r1 > r0:
            assert_gemm(got[r0:r1], ref[r0:r1], g[r0:r1], w[e], N, f"expert {e}")
    _no_device_error()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ci", range(len(GROUPED_COUNTS)))
def test_grouped_wgrad(fmt, ci, kernel, monkeypatch):
    _select_kernel(monkeypatch, kernel)
    counts = GROUPED_COUNTS[ci]
    S, N, K = sum(counts) + 9, 200, 352
    E = len(counts)
    offsets = synth.offsets_from_counts(counts)
    X = synth.make_packed(fmt, 1, S, K, 1.0, seed=40 + ci, device="cpu")
    G = _grad(S, N, 41 + ci)
    if offsets[-1] < S:
        G[int(offsets[-1]):] = float("nan")       # never read
    out = bsq.grouped_wgrad(G.cuda(), X.to("cuda"), torch.from_numpy(offsets).cuda(), E)
    torch.cuda.synchronize()
    got = bf16_vals(out)
    x = oracle_deq(X)[0]
    g = bf16_vals(G)
    ref = Gm.grouped_wgrad(g, x, offsets, E)
    for e in range(E):
        r0, r1 = Gm.expert_rows(offsets, e)
        if r1 == r0:
            assert (got[e] == 0).all(), f"empty expert {e} not zero"
        else:
            assert_gemm(got[e], ref[e], g[r0:r1], x[r0:r1], r1 - r0, f"expert {e}")
    _no_device_error()


def test_single_expert_grouped_equals_linear_bitwise():
    N, K, S = 256, 384, 333
    W = synth.make_packed(synth.FMT_MXFP4, 1, N, K, 1.0, seed=50, device="cpu").to("cuda")
    G = _grad(S, N, 51).cuda()
    a = bsq.linear_dgrad(G, W)
    b = bsq.grouped_dgrad(G, W, torch.tensor([S], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bad_offsets_are_reported_not_written():
    N, K, S = 128, 256, 64
    W = synth.make_packed(synth.FMT_FP8, 2, N, K, 1.0, seed=60, device="cpu").to("cuda")
    G = _grad(S, N, 61).cuda()
    out = torch.full((S, K), 7.0, dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G, W, torch.tensor([40, 20], dtype=torch.int32, device="cuda"), out=out)
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_ERR_INVALID_ARG and code == 2
    assert (out.float() == 7.0).all()
    _no_device_error()


def test_config1_full():
    c = synth.make_config(1, device="cpu")
    G, W, X = c["G"], c["W"], c["X"]
    gx = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    gw = bsq.linear_wgrad(G.cuda(), X.to("cuda"))
    torch.cuda.synchronize()
    g = bf16_vals(G)
    w = oracle_deq(W)[0]
    x = oracle_deq(X)[0]
    assert_gemm(bf16_vals(gx), Gm.dgrad(g, w), g, w, c["N"], "config1 dgrad")
    assert_gemm(bf16_vals(gw), Gm.wgrad(g, x), g, x, c["M"], "config1 wgrad")


def test_repeat_runs_are_bitwise_identical():
    W = synth.make_packed(synth.FMT_NVFP4, 1, 512, 768, 0.02, seed=70, device="cpu").to("cuda")
    G = _grad(1000, 512, 71, 1e-2).cuda()
    a = bsq.linear_dgrad(G, W)
    b = bsq.linear_dgrad(G, W)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
