"""Mutation smoke for the oracle pins: a mistake planted in the oracle (on the CPU)
must make at least one pin fail.  Mirrors the mutation testing described in MSLK
PR #393's test plan (an injected backward error must fail the suite)."""

import numpy as np
import pytest

import oracle.dequant as D
import oracle.formats as F
import oracle.gemm as Gm
import tests.test_oracle_dequant as TD
import tests.test_oracle_formats as TF
import tests.test_oracle_gemm as TG


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_swapped_nibbles_are_caught(monkeypatch):
    def swapped(packed, cols):
        packed = np.asarray(packed, dtype=np.uint8)
        codes = np.empty(packed.shape[:-1] + (cols,), dtype=np.uint8)
        codes[..., 0::2] = packed >> 4
        codes[..., 1::2] = packed & 0x0F
        return codes
    monkeypatch.setattr(D, "unpack_fp4", swapped)
    assert _fails(TD.test_fp4_nibble_order)
    assert _fails(TD.test_mxfp4_against_torch, "random")


def test_wrong_fp8_block_is_caught(monkeypatch):
    monkeypatch.setattr(D, "FP8_BLOCK", 64)
    assert _fails(TD.test_fp8_linear_example_shape_from_page)


def test_wrong_mx_block_is_caught(monkeypatch):
    monkeypatch.setattr(D, "MX_BLOCK", 16)
    assert _fails(TD.test_scale_block_indexing_mxfp4_and_nvfp4)


def test_skipped_scale_rounding_is_caught(monkeypatch):
    real = D.bf16_round
    calls = {"n": 0}

    def skip_second(x):           # drops the BF16 cast of the scale (second call per dequant)
        calls["n"] += 1
        return np.asarray(x, dtype=np.float64) if calls["n"] % 3 == 1 else real(x)
    monkeypatch.setattr(D, "bf16_round", skip_second)
    assert _fails(TD.test_fp8_all_codes_ragged_shapes, 200, 300)


def test_e4m3_bias_error_is_caught(monkeypatch):
    monkeypatch.setattr(F, "E4M3_TABLE", F.E4M3_TABLE * 2.0)
    assert _fails(TF.test_e4m3_table_matches_torch_float8)


def test_transposed_wgrad_is_caught(monkeypatch):
    monkeypatch.setattr(Gm, "wgrad", lambda g, x: Gm.as_f64(x).T @ Gm.as_f64(g))
    assert _fails(TG.test_dgrad_wgrad_brute_force, 3)


def test_grouped_off_by_one_is_caught(monkeypatch):
    def shifted(offsets, e):
        offsets = np.asarray(offsets, dtype=np.int64)
        r0 = 0 if e == 0 else int(offsets[e - 1]) + 1
        return r0, int(offsets[e])
    monkeypatch.setattr(Gm, "expert_rows", shifted)
    assert _fails(TG.test_grouped_dgrad_equals_block_diagonal_dense)


def test_per_tensor_scale_of_the_wrong_expert_is_caught(monkeypatch):
    real = D.scale_values

    def first_expert_only(fmt, scale, tensor_scale, batch, rows, cols):
        if fmt == D.FMT_FP8_TENSOR:
            s = np.asarray(scale, dtype=np.float32).astype(np.float64).reshape(batch)
            return np.broadcast_to(np.full((batch, 1, 1), s[0]), (batch, rows, cols))
        return real(fmt, scale, tensor_scale, batch, rows, cols)
    monkeypatch.setattr(D, "scale_values", first_expert_only)
    assert _fails(TD.test_fp8_per_tensor_scale_matches_page_recipe, "random")


def test_untransposed_forward_is_caught(monkeypatch):
    monkeypatch.setattr(Gm, "forward", lambda x, w: Gm.as_f64(w) @ Gm.as_f64(x).T)
    assert _fails(TG.test_forward_brute_force, 3)


def test_e5m2_rounding_half_up_is_caught(monkeypatch):
    import tests.test_oracle_quantize as TQ
    real_rint = np.rint

    class HalfUp:                       # np.rint replaced by round-half-away inside e5m2_round
        def __getattr__(self, name):
            if name == "rint":
                return lambda a: np.floor(np.asarray(a) + 0.5)
            return getattr(np, name)
    monkeypatch.setattr(F, "np", HalfUp())
    assert _fails(TQ.test_e5m2_round_ties_to_even_at_every_midpoint)
    assert real_rint is np.rint


def test_e5m2_bias_error_is_caught(monkeypatch):
    import tests.test_oracle_quantize as TQ
    monkeypatch.setattr(F, "E5M2_TABLE", F.E5M2_TABLE * 2.0)
    assert _fails(TQ.test_e5m2_table_matches_torch_float8)


def test_amax_without_abs_is_caught(monkeypatch):
    import oracle.quantize as Q
    import tests.test_oracle_quantize as TQ

    def signed_amax(g):
        g = np.asarray(g, dtype=np.float64)
        return float(max(F.fp32_round(np.max(g)), F.fp32_round(Q.AMAX_FLOOR)))
    monkeypatch.setattr(Q, "amax_f32", signed_amax)
    assert _fails(TQ.test_quantize_largest_element_lands_on_the_maximum)


def test_step_from_the_e4m3_maximum_is_caught(monkeypatch):
    import oracle.quantize as Q
    import tests.test_oracle_quantize as TQ
    monkeypatch.setattr(Q, "E5M2_MAX", F.E4M3_MAX)
    assert _fails(TQ.test_quantize_matches_the_page_recipe_in_torch, 1.0)
