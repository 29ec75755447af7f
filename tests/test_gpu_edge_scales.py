"""The fused dequant prologue of every GEMM entry point, pinned bit for bit on edge scales.

The GEMM parity tests draw quantized N(0, s) operands, whose scales all take the decode's
fast path (one BF16 multiply).  Here the packed operand is `synth.random_codes`: uniform
code bytes with scales that force the other paths of the prologue --

  * "finite": E8M0 bytes up to 200, float32 scale_inv with full mantissas from 2^-137 to
    2^117, NVFP4 tensor scales from 1e-30 to 1e30 (combined scales that are not BF16
    numbers, or are subnormal, or overflow the fast path's scaled form), every decoded
    value finite;
  * "nan": NaN codes and NaN scales.

grad_out is one-hot along the contraction, so each output element is one product 1 * v
plus exact zeros: the result is the oracle's dequantized element v itself (transformers
PR #50031 `_dequantize_fp8_weight` and MSLK PR #393 "Implementation Method": the product
of grad_out with the dequantized BF16 operand), and the comparison is on BF16 bits.  With
NaN or infinite values in the contraction the IEEE rules decide the element: a column
holding a NaN anywhere, or an infinity in a row the one-hot does not pick (0 * inf), is
NaN; those are compared as a NaN class.  Zeros compare without their sign (the sign of a
sum of signed zeros is not fixed by the method), and a value below the FP32 normal range
may come back as zero (the tensor core's FP32 accumulator) -- every other bit must match.
"""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import formats as F
from tests._util import oracle_deq

pytestmark = pytest.mark.gpu

PACKED = [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR]
KINDS = ["finite", "nan"]
FP32_TINY = 2.0 ** -126


def expected_one_hot(vals, picks):
    """vals: float64 [R, C] (the contraction rows); picks: row index per output row.
    Output row i = vals[picks[i]] under IEEE NaN / infinity rules for 1*v + sum(0*v')."""
    nan_col = np.isnan(vals).any(axis=0)
    inf = np.isinf(vals)
    inf_count = inf.sum(axis=0)
    rows = vals[picks]
    poisoned = nan_col[None, :] | ((inf_count[None, :] - inf[picks]) > 0)
    return np.where(poisoned, np.nan, rows)


def assert_bits(out_t, expected, what):
    got = synth.bf16_numpy(out_t).astype(np.uint16)
    gv = F.bf16_from_bits(got)
    en = np.isnan(expected)
    gn = np.isnan(gv)
    assert np.array_equal(gn, en), f"{what}: NaN class differs at {np.argwhere(gn != en)[:5].tolist()}"
    e = expected[~en]
    g = gv[~en]
    gb = got[~en]
    eb = F.bf16_bits(e)
    same = (gb == eb) | ((e == 0) & (g == 0))
    flushed = (~same) & (np.abs(e) < FP32_TINY) & (g == 0)
    bad = ~(same | flushed)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements differ, e.g. got {g[bad][:4]} "
                           f"expected {e[bad][:4]}")


def _one_hot_rows(n_rows, width, seed):
    """grad_out [n_rows, width] with one 1.0 per row; returns (tensor, picks)."""
    rng = np.random.default_rng(seed)
    picks = rng.integers(0, width, size=n_rows)
    picks[: min(n_rows, 3)] = [0, width - 1, width // 2][: min(n_rows, 3)]
    G = torch.zeros((n_rows, width), dtype=torch.bfloat16)
    G[torch.arange(n_rows), torch.from_numpy(picks)] = 1.0
    return G, picks


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
def test_linear_dgrad_one_hot_edge_scales(fmt, kind):
    M, N, K = 70, 200, 384       # ragged contraction (N), three m-tiles (odd pair member past the end)
    W = synth.random_codes(fmt, 1, N, K, seed=300 + fmt, scale_kind=kind)
    G, picks = _one_hot_rows(M, N, 301)
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    assert_bits(out, expected_one_hot(oracle_deq(W)[0], picks), f"dgrad fmt={fmt} {kind}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


@pytest.mark.parametrize("short", ["0", "1"])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
@pytest.mark.parametrize("N", [136, 192])
def test_linear_wgrad_one_hot_edge_scales(fmt, kind, N, short, monkeypatch):
    monkeypatch.setenv("BSQ_GEMM_SHORT_TILES", short)
    M, K = 200, 384
    X = synth.random_codes(fmt, 1, M, K, seed=310 + fmt, scale_kind=kind)
    Gt, picks = _one_hot_rows(N, M, 311)      # grad_out^T: one token per output row n
    G = Gt.t().contiguous()
    out = bsq.linear_wgrad(G.cuda(), X.to("cuda"))
    torch.cuda.synchronize()
    assert_bits(out, expected_one_hot(oracle_deq(X)[0], picks), f"wgrad fmt={fmt} {kind} N={N}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


COUNTS = [3, 0, 70, 1, 130]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
def test_grouped_dgrad_one_hot_edge_scales(fmt, kind):
    N, K = 200, 384
    E = len(COUNTS)
    offs = synth.offsets_from_counts(COUNTS)
    S = int(offs[-1]) + 5
    W = synth.random_codes(fmt, E, N, K, seed=320 + fmt, scale_kind=kind)
    G, picks = _one_hot_rows(S, N, 321)
    out = torch.full((S, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G.cuda(), W.to("cuda"), torch.from_numpy(offs).cuda(), out=out)
    torch.cuda.synchronize()
    w = oracle_deq(W)
    for e in range(E):
        r0 = 0 if e == 0 else int(offs[e - 1])
        r1 = int(offs[e])
        if r1 > r0:
            assert_bits(out[r0:r1], expected_one_hot(w[e], picks[r0:r1]), f"grouped dgrad e={e} fmt={fmt} {kind}")
    assert torch.isnan(out[int(offs[-1]):].float()).all()
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


@pytest.mark.parametrize("short", ["0", "1"])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
def test_grouped_wgrad_one_hot_edge_scales(fmt, kind, short, monkeypatch):
    monkeypatch.setenv("BSQ_GEMM_SHORT_TILES", short)
    N, K = 136, 384
    E = len(COUNTS)
    offs = synth.offsets_from_counts(COUNTS)
    S = int(offs[-1]) + 5
    X = synth.random_codes(fmt, 1, S, K, seed=330 + fmt, scale_kind=kind)
    rng = np.random.default_rng(331)
    G = torch.zeros((S, N), dtype=torch.bfloat16)
    G[int(offs[-1]):] = float("nan")            # rows past offsets[E-1] are never read
    picks = {}
    for e in range(E):
        r0 = 0 if e == 0 else int(offs[e - 1])
        r1 = int(offs[e])
        if r1 > r0:
            t = rng.integers(r0, r1, size=N)
            G[torch.from_numpy(t), torch.arange(N)] = 1.0
            picks[e] = t - r0
    out = bsq.grouped_wgrad(G.cuda(), X.to("cuda"), torch.from_numpy(offs).cuda(), E)
    torch.cuda.synchronize()
    x = oracle_deq(X)[0]
    for e in range(E):
        r0 = 0 if e == 0 else int(offs[e - 1])
        r1 = int(offs[e])
        if r1 == r0:
            assert (out[e].float() == 0).all().item(), f"empty expert {e}"
        else:
            assert_bits(out[e], expected_one_hot(x[r0:r1], picks[e]), f"grouped wgrad e={e} fmt={fmt} {kind}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


# ---- the small-M kernels (their own decode): M <= 16 linear dgrad, decode-sized grouped dgrad


@pytest.mark.parametrize("M", [1, 9, 16])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
def test_small_m_dgrad_one_hot_edge_scales(fmt, kind, M):
    N, K = 200, 384       # ragged contraction over three 64-row chunks, three 128-column slabs
    W = synth.random_codes(fmt, 1, N, K, seed=340 + fmt, scale_kind=kind)
    G, picks = _one_hot_rows(M, N, 341 + M)
    out = bsq.linear_dgrad(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    assert_bits(out, expected_one_hot(oracle_deq(W)[0], picks), f"small-M dgrad M={M} fmt={fmt} {kind}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4])   # the formats it takes
def test_small_m_noalloc_one_hot_edge_scales(fmt, kind):
    M, N, K = 12, 200, 384
    W = synth.random_codes(fmt, 1, N, K, seed=350 + fmt, scale_kind=kind)
    G, picks = _one_hot_rows(M, N, 351)
    out = bsq.linear_dgrad_smallm_noalloc(G.cuda(), W.to("cuda"))
    torch.cuda.synchronize()
    assert_bits(out, expected_one_hot(oracle_deq(W)[0], picks), f"noalloc small-M dgrad fmt={fmt} {kind}")
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


DECODE_COUNTS = [3, 0, 20, 1, 30]   # 54 rows in all: the decode-sized grouped path


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", PACKED)
def test_grouped_decode_one_hot_edge_scales(fmt, kind):
    N, K = 200, 384
    E = len(DECODE_COUNTS)
    offs = synth.offsets_from_counts(DECODE_COUNTS)
    S = int(offs[-1]) + 5
    W = synth.random_codes(fmt, E, N, K, seed=360 + fmt, scale_kind=kind)
    G, picks = _one_hot_rows(S, N, 361)
    out = torch.full((S, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    bsq.grouped_dgrad(G.cuda(), W.to("cuda"), torch.from_numpy(offs).cuda(), out=out)
    torch.cuda.synchronize()
    w = oracle_deq(W)
    for e in range(E):
        r0 = 0 if e == 0 else int(offs[e - 1])
        r1 = int(offs[e])
        if r1 > r0:
            assert_bits(out[r0:r1], expected_one_hot(w[e], picks[r0:r1]), f"decode dgrad e={e} fmt={fmt} {kind}")
    assert torch.isnan(out[int(offs[-1]):].float()).all()
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)
