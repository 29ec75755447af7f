"""Pins for the oracle's float64 products (CPU only): exact rational brute force,
closed forms from the pages' worked examples, and the grouped form rebuilt as one
block-diagonal dense product."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import dequant as D
from oracle import formats as F
from oracle import gemm as Gm

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def _frac_matmul(a, b):
    n, k = len(a), len(a[0])
    m = len(b[0])
    return [[sum((Fraction(a[i][t]) * Fraction(b[t][j]) for t in range(k)), Fraction(0)) for j in range(m)]
            for i in range(n)]


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_dgrad_wgrad_brute_force(n):
    rng = np.random.default_rng(n)
    # dyadic values (integers / 64): every product and sum is exact in float64
    g = rng.integers(-40, 40, size=(n, n + 1)) / 64.0
    w = rng.integers(-40, 40, size=(n + 1, n + 2)) / 64.0
    x = rng.integers(-40, 40, size=(n, n + 2)) / 64.0
    exp_d = _frac_matmul(g.tolist(), w.tolist())
    got_d = Gm.dgrad(g, w)
    assert all(got_d[i][j] == exp_d[i][j] for i in range(n) for j in range(n + 2))
    gt = g.T.tolist()
    exp_w = _frac_matmul(gt, x.tolist())
    got_w = Gm.wgrad(g, x)
    assert got_w.shape == (n + 1, n + 2)
    assert all(got_w[i][j] == exp_w[i][j] for i in range(n + 1) for j in range(n + 2))


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_forward_brute_force(n):
    """Y = X @ W^T against exact rational arithmetic (the contraction is over K, the axis X
    and W both store contiguously)."""
    rng = np.random.default_rng(100 + n)
    x = rng.integers(-40, 40, size=(n, n + 3)) / 64.0
    w = rng.integers(-40, 40, size=(n + 1, n + 3)) / 64.0
    exp = _frac_matmul(x.tolist(), w.T.tolist())
    got = Gm.forward(x, w)
    assert got.shape == (n, n + 1)
    assert all(got[i][j] == exp[i][j] for i in range(n) for j in range(n + 1))


def test_forward_closed_forms():
    """One-hot rows of X pick columns of W: Y[i, j] = W[j, k_i]; and the forward is the
    transpose of a dgrad against the other operand: (X W^T)^T = W X^T."""
    rng = np.random.default_rng(7)
    w = rng.standard_normal((6, 9))
    ks = [0, 4, 8]
    x = np.zeros((3, 9))
    x[range(3), ks] = 1.0
    np.testing.assert_array_equal(Gm.forward(x, w), w[:, ks].T)
    xr = rng.standard_normal((4, 9))
    np.testing.assert_allclose(Gm.forward(xr, w).T, Gm.dgrad(w, xr.T), rtol=0, atol=1e-12)


def test_bf16_bit_inputs_are_decoded():
    bits = np.array([[0x3F80, 0xC000]], dtype=np.uint16)   # 1.0, -2.0
    w = np.array([[3.0], [0.5]])
    assert Gm.dgrad(bits, w)[0, 0] == 2.0


def _fp8_weight(N, K, seed, grid=None):
    g = torch.Generator().manual_seed(seed)
    codes = torch.randn(N, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if grid is None:
        grid = (torch.rand(-(-N // 128), -(-K // 128), generator=g) + 0.5).numpy().astype(np.float32)
    return codes, grid


def test_ones_grad_gives_column_sums_page_example():
    ex = GOLDEN["fp8_linear_example"]
    N, K = ex["out_features"], ex["in_features"]
    codes, grid = _fp8_weight(N, K, 2)
    w = D.dequant_values(D.FMT_FP8, codes, grid, None, 1, N, K)[0]
    tokens = int(np.prod(ex["input_shape"][:-1]))
    ones = np.ones((tokens, N))
    gx = Gm.dgrad(ones, w)
    colsum = np.array([sum(Fraction(v) for v in w[:, k]) for k in range(K)], dtype=object)
    for t in range(tokens):
        assert all(gx[t, k] == float(colsum[k]) for k in range(K))


def test_grouped_ones_grad_page_example():
    ex = GOLDEN["fp8_grouped_example"]
    E, (N, K) = ex["groups"], ex["per_group_weight"]
    tokens = ex["input_shape"][0]
    codes, grid = _fp8_weight(E * N, K, 3)
    w = D.dequant_values(D.FMT_FP8, codes.reshape(E, N, K), grid.reshape(E, N // 128, K // 128), None, E, N, K)
    offsets = np.array([tokens * (e + 1) for e in range(E)], dtype=np.int32)
    gx = Gm.grouped_dgrad(np.ones((tokens * E, N)), w, offsets)
    for e in range(E):
        np.testing.assert_array_equal(gx[e * tokens:(e + 1) * tokens], np.tile(w[e].sum(axis=0), (tokens, 1)))


def test_one_hot_rows_select_weight_rows_exactly():
    N, K = 256, 384
    codes, grid = _fp8_weight(N, K, 4)
    w = D.dequant_values(D.FMT_FP8, codes, grid, None, 1, N, K)[0]
    idx = np.array([0, 17, 255, 128])
    g = np.zeros((len(idx), N))
    g[np.arange(len(idx)), idx] = 1.0
    np.testing.assert_array_equal(Gm.dgrad(g, w), w[idx])
    x = w.T[:, :N].copy()           # any [M, K'] operand
    np.testing.assert_array_equal(Gm.wgrad(np.zeros((K, N)), np.ones((K, 5))), np.zeros((N, 5)))
    assert x.shape[1] == N


def _routing(S, E, seed, empty=()):
    rng = np.random.default_rng(seed)
    counts = rng.multinomial(S, np.ones(E) / E)
    for e in empty:
        counts[e] = 0
    return np.cumsum(counts).astype(np.int32)


def test_grouped_dgrad_equals_block_diagonal_dense():
    S, E, N, K = 50, 4, 12, 7
    rng = np.random.default_rng(0)
    g = rng.standard_normal((S, N))
    w = rng.standard_normal((E, N, K))
    offsets = _routing(S - 3, E, 1, empty=(1,))   # last 3 rows belong to no expert
    big_g = np.zeros((S, E * N))
    for e in range(E):
        r0, r1 = Gm.expert_rows(offsets, e)
        big_g[r0:r1, e * N:(e + 1) * N] = g[r0:r1]
    ref = big_g @ w.reshape(E * N, K)
    out = Gm.grouped_dgrad(g, w, offsets)
    used = int(offsets[-1])
    np.testing.assert_allclose(out[:used], ref[:used], rtol=1e-12, atol=1e-12)
    assert np.isnan(out[used:]).all()


def test_grouped_wgrad_equals_block_diagonal_dense_and_empty_is_zero():
    S, E, N, K = 60, 5, 9, 11
    rng = np.random.default_rng(1)
    g = rng.standard_normal((S, N))
    x = rng.standard_normal((S, K))
    offsets = _routing(S - 4, E, 2, empty=(0, 4))
    g[int(offsets[-1]):] = np.nan                   # tail rows are never read
    big_x = np.zeros((S, E * K))
    for e in range(E):
        r0, r1 = Gm.expert_rows(offsets, e)
        big_x[r0:r1, e * K:(e + 1) * K] = x[r0:r1]
    gg = np.nan_to_num(g)
    ref = (gg.T @ big_x).reshape(N, E, K).transpose(1, 0, 2)
    out = Gm.grouped_wgrad(g, x, offsets, E)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert (out[0] == 0).all() and (out[4] == 0).all()


def test_single_expert_equals_linear():
    rng = np.random.default_rng(5)
    g = rng.standard_normal((33, 10))
    w = rng.standard_normal((1, 10, 6))
    x = rng.standard_normal((33, 6))
    off = np.array([33], dtype=np.int32)
    np.testing.assert_array_equal(Gm.grouped_dgrad(g, w, off), Gm.dgrad(g, w[0]))
    np.testing.assert_array_equal(Gm.grouped_wgrad(g, x, off, 1)[0], Gm.wgrad(g, x))


def test_tolerance_check_catches_planted_errors():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((64, 256))
    b = rng.standard_normal((256, 32))
    ref = a @ b
    bound = Gm.tolerance(256, a, b)
    ok, _, _ = Gm.check(ref + 1e-6, ref, bound)
    assert ok
    bad = ref.copy()
    bad[3, 4] += 5 * bound                          # one wrong element
    assert not Gm.check(bad, ref, bound)[0]
    dropped = a[:, :-1] @ b[:-1]                    # a dropped term of the contraction
    assert not Gm.check(dropped, ref, bound)[0]
    assert not Gm.check(a @ b[:, ::-1], ref, bound)[0]   # permuted output columns
    assert not Gm.check(np.zeros_like(ref), np.zeros_like(ref) + 1, 0.0)[0]
    assert Gm.check(np.zeros((2, 2)), np.zeros((2, 2)), 0.0)[0]


def test_output_rounding_allowance_is_half_an_ulp():
    # one-term products: the only error a correct BF16 result can have is its own rounding
    rng = np.random.default_rng(8)
    from oracle.formats import bf16_round
    a = bf16_round(rng.standard_normal((50, 1)) * 3)
    b = bf16_round(rng.standard_normal((1, 60)) * 3)
    ref = a @ b
    out = bf16_round(ref)
    assert Gm.check(out, ref, Gm.tolerance(1, a, b))[0]
    worse = out + np.sign(ref) * np.abs(ref) * 2.0 ** -7      # a full extra ulp-sized error
    assert not Gm.check(worse, ref, 0.0)[0]
