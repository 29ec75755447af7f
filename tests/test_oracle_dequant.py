"""Pins for the oracle's dequantization (CPU only).

The expected values are computed a second way with torch on the CPU, following the
transformers PR #50031 `_dequantize_fp8_weight` recipe (scale cast to BF16, grid
repeated per block and cropped, weight cast to BF16, product rounded to BF16) or,
for FP4, from the E2M1/E8M0/E4M3 values computed by torch's own float32/BF16
arithmetic.  A product of a BF16 code value and a BF16 scale is exact in float32,
so torch's float32-then-round path is a single nearest-even rounding as well.
"""

import json
import os

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import synth
from oracle import dequant as D
from oracle import formats as F

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def _torch_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _same_bits(got, ref):
    """Bit equality, every NaN pattern counted as one class."""
    gn, rn = F.bf16_is_nan_bits(got), F.bf16_is_nan_bits(ref)
    return np.array_equal(gn, rn) and np.array_equal(got[~gn], ref[~rn])


def _torch_fp8_dequant(codes_u8, scale_inv, rows, cols):
    """The page's recipe with torch ops: [rows, cols] BF16."""
    w = torch.from_numpy(codes_u8).view(torch.float8_e4m3fn).to(torch.bfloat16)
    s = torch.from_numpy(scale_inv).to(torch.bfloat16)
    s = s.repeat_interleave(128, dim=-2)[..., :rows, :].repeat_interleave(128, dim=-1)[..., :cols]
    return w * s


def _torch_fp8_tensor_dequant(codes_u8, scale_inv):
    """The page's recipe with block_size None, with torch ops: the scale cast to BF16 and
    broadcast (one per batch entry), the weight cast to BF16, product rounded to BF16."""
    w = torch.from_numpy(codes_u8).view(torch.float8_e4m3fn).to(torch.bfloat16)
    s = torch.from_numpy(np.asarray(scale_inv, dtype=np.float32)).to(torch.bfloat16)
    return w * s.reshape(-1, *([1] * (w.dim() - 1)))


@pytest.mark.parametrize("kind", ["random", "edge", "nan", "finite"])
def test_fp8_per_tensor_scale_matches_page_recipe(kind):
    """transformers PR #50031 `_dequantize_fp8_weight`, `block_size is None`: every code of a
    three-expert weight against the torch restatement of that branch."""
    p = synth.random_codes(synth.FMT_FP8_TENSOR, 3, 130, 96, seed=21, scale_kind=kind)
    d, s, _ = p.numpy()
    got = D.dequant_bits(D.FMT_FP8_TENSOR, d, s, None, 3, 130, 96)
    assert _same_bits(got, _torch_bits(_torch_fp8_tensor_dequant(d, s)))
    cols, rows = np.array([0, 17, 95]), np.array([0, 64, 129])
    full = D.dequant_values(D.FMT_FP8_TENSOR, d, s, None, 3, 130, 96)
    for b in range(3):
        np.testing.assert_array_equal(D.dequant_cols(D.FMT_FP8_TENSOR, d, s, None, 130, 96, cols, b, 3),
                                      full[b][:, cols])
        np.testing.assert_array_equal(D.dequant_rows(D.FMT_FP8_TENSOR, d, s, None, 130, 96, rows, b, 3),
                                      full[b][rows])


def test_fp8_per_tensor_scale_is_a_constant_block_grid():
    """One scale per tensor decodes exactly as 128x128 blocks that all hold that scale."""
    p = synth.random_codes(synth.FMT_FP8_TENSOR, 2, 300, 256, seed=22)
    d, s, _ = p.numpy()
    grid = np.repeat(s.reshape(2, 1, 1), 3, axis=1).repeat(2, axis=2).astype(np.float32)
    a = D.dequant_bits(D.FMT_FP8_TENSOR, d, s, None, 2, 300, 256)
    b = D.dequant_bits(D.FMT_FP8, d, grid, None, 2, 300, 256)
    assert _same_bits(a, b)


def test_fp8_linear_example_shape_from_page():
    ex = GOLDEN["fp8_linear_example"]
    N, K = ex["out_features"], ex["in_features"]
    g = torch.Generator().manual_seed(0)
    codes = torch.randn(N, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    grid = (torch.rand(*ex["scale_grid"], generator=g) + 0.5).numpy().astype(np.float32)
    assert grid.shape == (-(-N // 128), -(-K // 128))
    ref = _torch_bits(_torch_fp8_dequant(codes, grid, N, K))
    got = D.dequant_bits(D.FMT_FP8, codes, grid, None, 1, N, K).reshape(N, K)
    assert _same_bits(got, ref)


@pytest.mark.parametrize("rows,cols", [(200, 300), (1, 16), (129, 127), (384, 256)])
def test_fp8_all_codes_ragged_shapes(rows, cols):
    p = synth.random_codes(synth.FMT_FP8, 1, rows, cols, seed=rows * 7 + cols)
    d, s, _ = p.numpy()
    ref = _torch_bits(_torch_fp8_dequant(d[0], s[0], rows, cols))
    got = D.dequant_bits(D.FMT_FP8, d, s, None, 1, rows, cols).reshape(rows, cols)
    assert _same_bits(got, ref)


@pytest.mark.parametrize("kind", ["edge", "nan"])
def test_fp8_edge_and_nan_scales(kind):
    p = synth.random_codes(synth.FMT_FP8, 2, 256, 384, seed=11, scale_kind=kind)
    d, s, _ = p.numpy()
    got = D.dequant_bits(D.FMT_FP8, d, s, None, 2, 256, 384).reshape(2, 256, 384)
    for b in range(2):
        ref = _torch_bits(_torch_fp8_dequant(d[b], s[b], 256, 384))
        assert _same_bits(got[b], ref)


def test_fp8_grouped_example_is_per_expert_grid():
    ex = GOLDEN["fp8_grouped_example"]
    E, (N, K) = ex["groups"], ex["per_group_weight"]
    g = torch.Generator().manual_seed(1)
    codes = torch.randn(E * N, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    grid = (torch.rand(*ex["scale_grid"], generator=g) + 0.5).numpy().astype(np.float32)
    ref = _torch_bits(_torch_fp8_dequant(codes, grid, E * N, K)).reshape(E, N, K)
    got = D.dequant_bits(D.FMT_FP8, codes.reshape(E, N, K), grid.reshape(E, N // 128, K // 128), None, E, N, K)
    assert _same_bits(got.reshape(E, N, K), ref)


def _torch_fp4_values(packed, cols):
    """E2M1 values via bit fields computed by torch integer ops (independent of the oracle table)."""
    p = torch.from_numpy(packed).to(torch.int32)
    codes = torch.stack([p & 0xF, p >> 4], dim=-1).reshape(*p.shape[:-1], cols)
    sign = torch.where((codes & 8) != 0, -1.0, 1.0)
    e = (codes >> 1) & 3
    m = (codes & 1).to(torch.float32)
    mag = torch.where(e == 0, m * 0.5, (1 + m / 2) * torch.pow(2.0, (e - 1).to(torch.float32)))
    return sign * mag


def test_fp4_nibble_order():
    packed = np.array([[[0x21, 0x8F]]], dtype=np.uint8)   # codes 1,2 then 0xF,0x8
    scale = np.array([[[127]]], dtype=np.uint8)
    cols = 32
    packed = np.concatenate([packed, np.zeros((1, 1, 14), np.uint8)], axis=-1)
    v = D.dequant_values(D.FMT_MXFP4, packed, scale, None, 1, 1, cols)[0, 0]
    assert v[0] == 0.5 and v[1] == 1.0 and v[2] == -6.0 and v[3] == 0.0 and np.signbit(v[3])


@pytest.mark.parametrize("kind", ["random", "edge", "nan"])
def test_mxfp4_against_torch(kind):
    B, R, C = 2, 96, 320
    p = synth.random_codes(synth.FMT_MXFP4, B, R, C, seed=5, scale_kind=kind)
    d, s, _ = p.numpy()
    vals = _torch_fp4_values(d, C)
    sc = torch.from_numpy(s).to(torch.float64)
    sc = torch.where(sc == 255, torch.nan, torch.pow(2.0, sc - 127)).repeat_interleave(32, dim=-1)
    ref = _torch_bits((vals.to(torch.float32) * sc.to(torch.float32)).to(torch.bfloat16))
    got = D.dequant_bits(D.FMT_MXFP4, d, s, None, B, R, C).reshape(B, R, C)
    # float32 holds every product except overflow, where both sides give infinity
    assert _same_bits(got, ref)


@pytest.mark.parametrize("kind", ["random", "edge", "nan"])
def test_nvfp4_against_torch(kind):
    B, R, C = 3, 40, 144
    p = synth.random_codes(synth.FMT_NVFP4, B, R, C, seed=9, scale_kind=kind)
    d, s, ts = p.numpy()
    vals = _torch_fp4_values(d, C).to(torch.bfloat16)
    blk = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float32)
    comb = (blk * torch.from_numpy(ts).view(B, 1, 1)).to(torch.bfloat16)   # one float32 product, then BF16
    ref = _torch_bits(vals * comb.repeat_interleave(16, dim=-1))
    got = D.dequant_bits(D.FMT_NVFP4, d, s, ts, B, R, C).reshape(B, R, C)
    assert _same_bits(got, ref)


def test_scale_block_indexing_mxfp4_and_nvfp4():
    R, C = 3, 64
    packed = np.full((1, R, C // 2), 0x22, dtype=np.uint8)    # every code = 1.0
    s_mx = np.arange(R * C // 32, dtype=np.uint8).reshape(1, R, C // 32) + 120
    v = D.dequant_values(D.FMT_MXFP4, packed, s_mx, None, 1, R, C)[0]
    for r in range(R):
        for c in range(C):
            assert v[r, c] == 2.0 ** (int(s_mx[0, r, c // 32]) - 127)
    s_nv = (np.arange(R * C // 16, dtype=np.uint8).reshape(1, R, C // 16) + 0x30)
    ts = np.array([0.25], dtype=np.float32)
    v = D.dequant_values(D.FMT_NVFP4, packed, s_nv, ts, 1, R, C)[0]
    for r in range(R):
        for c in range(C):
            assert v[r, c] == F.bf16_round(F.E4M3_TABLE[s_nv[0, r, c // 16]] * 0.25)


def test_partial_decoders_agree_with_full():
    for fmt, fid in [(D.FMT_FP8, synth.FMT_FP8), (D.FMT_MXFP4, synth.FMT_MXFP4), (D.FMT_NVFP4, synth.FMT_NVFP4)]:
        p = synth.random_codes(fid, 2, 260, 192, seed=4)
        d, s, ts = p.numpy()
        full = D.dequant_values(fmt, d, s, ts, 2, 260, 192)
        cols = np.array([0, 5, 31, 32, 100, 191])
        rows = np.array([0, 1, 127, 128, 259])
        for b in range(2):
            np.testing.assert_array_equal(D.dequant_cols(fmt, d, s, ts, 260, 192, cols, b, 2), full[b][:, cols])
            np.testing.assert_array_equal(D.dequant_rows(fmt, d, s, ts, 260, 192, rows, b, 2), full[b][rows])
