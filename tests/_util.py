"""Shared helpers for the parity tests: run the oracle on the same seeded inputs the
CUDA library gets, and apply the acceptance bounds."""

import numpy as np
import torch

from block_scaled_gemm_fp8_gb300 import synth
from oracle import dequant as D
from oracle import formats as F
from oracle import gemm as Gm

ORACLE_FMT = {synth.FMT_BF16: D.FMT_BF16, synth.FMT_FP8: D.FMT_FP8, synth.FMT_MXFP4: D.FMT_MXFP4,
              synth.FMT_NVFP4: D.FMT_NVFP4}


def oracle_deq(p):
    """float64 [batch, rows, cols] dequantized values of a Packed operand (any device)."""
    d, s, ts = p.numpy()
    return D.dequant_values(ORACLE_FMT[p.fmt], d, s, ts, p.batch, p.rows, p.cols)


def oracle_deq_bits(p):
    d, s, ts = p.numpy()
    return D.dequant_bits(ORACLE_FMT[p.fmt], d, s, ts, p.batch, p.rows, p.cols)


def bf16_vals(t):
    """float64 values of a BF16 torch tensor."""
    return F.bf16_from_bits(synth.bf16_numpy(t))


def same_bits(got, ref):
    gn, rn = F.bf16_is_nan_bits(got), F.bf16_is_nan_bits(ref)
    if not np.array_equal(gn, rn):
        return False
    return np.array_equal(got[~gn], ref[~rn])


def assert_gemm(out, ref, a, b, kc, what=""):
    """The acceptance rule: |err| <= 2e-2 sqrt(Kc) rms(A) rms(B) elementwise and relative
    Frobenius error <= 5e-3 against the float64 oracle (A, B: the BF16 operands)."""
    bound = Gm.tolerance(kc, a, b)
    ok, max_err, rel = Gm.check(out, ref, bound)
    assert ok, f"{what}: max|err|={max_err:.4g} bound={bound:.4g} relF={rel:.3g}"
    return max_err, rel


def to_dev(p, device="cuda"):
    return p.to(device)


def routing_offsets(counts):
    return synth.offsets_from_counts(counts)
