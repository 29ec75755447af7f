"""Shared helpers for the parity tests: run the oracle on the same seeded inputs the
CUDA library gets, and apply the acceptance bounds."""

import numpy as np
import torch

from block_scaled_gemm_fp8_gb300 import synth
from oracle import dequant as D
from oracle import formats as F
from oracle import gemm as Gm

ORACLE_FMT = {synth.FMT_BF16: D.FMT_BF16, synth.FMT_FP8: D.FMT_FP8, synth.FMT_MXFP4: D.FMT_MXFP4,
              synth.FMT_NVFP4: D.FMT_NVFP4, synth.FMT_FP8_TENSOR: D.FMT_FP8_TENSOR,
              synth.FMT_E5M2_TENSOR: D.FMT_E5M2_TENSOR}


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


def block_cols(K, per_block, seed):
    """Column indices covering every 128-column block of an output with K columns (one
    m-tile of the GEMM kernels): the block's first and last column plus per_block - 2
    seeded ones, so that a wrong block of any CTA is seen."""
    rng = np.random.default_rng(seed)
    cols = []
    for b0 in range(0, K, 128):
        b1 = min(K, b0 + 128)
        pick = {b0, b1 - 1}
        if b1 - b0 > 2 and per_block > 2:
            pick |= set(rng.choice(np.arange(b0 + 1, b1 - 1), size=min(per_block - 2, b1 - b0 - 2),
                                   replace=False).tolist())
        cols.extend(sorted(pick))
    return np.array(cols, dtype=np.int64)


def deq_cols(p, cols, b=0):
    """float64 [rows, len(cols)]: the oracle's dequantized columns `cols` of batch entry b."""
    d, s, ts = p.numpy()
    return D.dequant_cols(ORACLE_FMT[p.fmt], d, s, ts, p.rows, p.cols, cols, b, p.batch)


def run_config(c, outs=None, fused=True):
    """Launch every op of a workload (bsq_*), into `outs` when given; returns the outputs.
    A linear workload runs as one bsq_linear_backward call (as bench.py times it) unless
    fused is False, which calls bsq_linear_dgrad and bsq_linear_wgrad."""
    from block_scaled_gemm_fp8_gb300 import bsq
    outs = {} if outs is None else outs
    if not c["grouped"] and fused:
        outs["dgrad"], outs["wgrad"] = bsq.linear_backward(c["G"], c["W"], c["X"], grad_x=outs.get("dgrad"),
                                                           grad_w=outs.get("wgrad"))
    elif not c["grouped"]:
        outs["dgrad"] = bsq.linear_dgrad(c["G"], c["W"], out=outs.get("dgrad"))
        outs["wgrad"] = bsq.linear_wgrad(c["G"], c["X"], out=outs.get("wgrad"))
    else:
        if "offsets_dev" not in c:
            c["offsets_dev"] = torch.from_numpy(c["offsets"]).to(c["G"].device)
        outs["grouped_dgrad"] = bsq.grouped_dgrad(c["G"], c["W"], c["offsets_dev"], out=outs.get("grouped_dgrad"))
        if c["X"] is not None:
            outs["grouped_wgrad"] = bsq.grouped_wgrad(c["G"], c["X"], c["offsets_dev"], c["E"],
                                                      out=outs.get("grouped_wgrad"))
    torch.cuda.synchronize()
    return outs


def check_config_sampled(c, outs, cols):
    """Check the outputs of a workload (any of dgrad, wgrad, small_m, grouped_dgrad,
    grouped_wgrad) against the float64 oracle on output columns `cols`, every row."""
    N = c["N"]
    if "small_m" in outs:
        w = deq_cols(c["W"], cols)
        gs = bf16_vals(c["G_small"])
        assert_gemm(bf16_vals(outs["small_m"][:, cols]), gs @ w, gs, w, N, f"{c['name']} small-M dgrad")
        return
    g = bf16_vals(c["G"])
    if not c["grouped"]:
        if "dgrad" in outs:
            w = deq_cols(c["W"], cols)
            assert_gemm(bf16_vals(outs["dgrad"][:, cols]), g @ w, g, w, N, f"{c['name']} dgrad")
        if "wgrad" in outs:
            x = deq_cols(c["X"], cols)
            assert_gemm(bf16_vals(outs["wgrad"][:, cols]), g.T @ x, g, x, c["M"], f"{c['name']} wgrad")
        return
    offs = c["offsets"]
    gx = bf16_vals(outs["grouped_dgrad"][:, cols]) if "grouped_dgrad" in outs else None
    gw = outs.get("grouped_wgrad")
    x = deq_cols(c["X"], cols) if gw is not None else None
    gws = bf16_vals(gw[:, :, cols]) if gw is not None else None
    for e in range(c["E"]):
        r0, r1 = Gm.expert_rows(offs, e)
        if r1 == r0:
            if gws is not None:
                assert (gws[e] == 0).all(), f"empty expert {e} not zero"
            continue
        if gx is not None:
            w = deq_cols(c["W"], cols, e)
            assert_gemm(gx[r0:r1], g[r0:r1] @ w, g[r0:r1], w, N, f"{c['name']} dgrad e={e}")
        if gws is not None:
            xe = x[r0:r1]
            assert_gemm(gws[e], g[r0:r1].T @ xe, g[r0:r1], xe, r1 - r0, f"{c['name']} wgrad e={e}")
