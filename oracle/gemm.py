"""The two backward products in float64, dense and per expert (oracle; test infrastructure only).

  grad_X = grad_out @ W_bf16      (dgrad)  -- MSLK PR #393, "Implementation Method";
                                             transformers PR #50031, `FP8LinearFunction.backward`
  grad_W = grad_out^T @ X_bf16    (wgrad)  -- MSLK PR #393, "Implementation Method"
  Y      = X_bf16 @ W_bf16^T      (forward) -- the product those two are the gradients of

Grouped form (transformers PR #50031, `FP8GroupedMatmulFunction.backward`, and the
offsets built in `FP8GroupedLinear.forward`): ``offsets`` is an int32 array of E
cumulative END offsets with no leading zero, so expert e owns token rows
[offsets[e-1] (0 for e = 0), offsets[e]).  Rows at or beyond offsets[E-1] belong to
no expert: the grouped dgrad leaves them unwritten (the page's comment in
`fp8_grouped_mm_experts_forward`), and the grouped wgrad does not read them.

Operands are float64 arrays holding BF16 values (from :mod:`oracle.dequant` or a
BF16 bit pattern); numpy's float64 matrix product is the library primitive.
"""

import numpy as np

from .formats import bf16_from_bits


def as_f64(bits_or_values):
    a = np.asarray(bits_or_values)
    if a.dtype == np.uint16:
        return bf16_from_bits(a)
    return a.astype(np.float64)


def dgrad(grad_out, w):
    """grad_X[M,K] = grad_out[M,N] @ W[N,K]."""
    return as_f64(grad_out) @ as_f64(w)


def wgrad(grad_out, x):
    """grad_W[N,K] = grad_out[M,N]^T @ X[M,K]."""
    return as_f64(grad_out).T @ as_f64(x)


def forward(x, w):
    """Y[M,N] = X[M,K] @ W[N,K]^T -- the forward of the linear layer whose gradients dgrad and
    wgrad are (MSLK PR #393, Summary: the `mslk::f4f4bf16` ops multiply packed X and W; the
    backward the PR adds differentiates that product)."""
    return as_f64(x) @ as_f64(w).T


def expert_rows(offsets, e):
    offsets = np.asarray(offsets, dtype=np.int64)
    r0 = 0 if e == 0 else int(offsets[e - 1])
    return r0, int(offsets[e])


def grouped_dgrad(grad_out, w, offsets):
    """grad_X[S,K]: rows of expert e are grad_out[r0:r1] @ W[e]; rows >= offsets[E-1] are NaN.

    NaN marks "not written": the library must leave those rows as they were.
    """
    g = as_f64(grad_out)
    w = as_f64(w)
    E, _, K = w.shape
    out = np.full((g.shape[0], K), np.nan)
    for e in range(E):
        r0, r1 = expert_rows(offsets, e)
        out[r0:r1] = g[r0:r1] @ w[e]
    return out


def grouped_wgrad(grad_out, x, offsets, E):
    """grad_W[E,N,K]: grad_W[e] = grad_out[r0:r1]^T @ X[r0:r1]; an empty expert gives zeros."""
    g = as_f64(grad_out)
    x = as_f64(x)
    out = np.zeros((E, g.shape[1], x.shape[1]))
    for e in range(E):
        r0, r1 = expert_rows(offsets, e)
        out[e] = g[r0:r1].T @ x[r0:r1]
    return out


def rms(a):
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def tolerance(kc, a, b):
    """Elementwise bound 2e-2 * sqrt(Kc) * rms(A) * rms(B) for one product of contraction Kc."""
    return 2e-2 * np.sqrt(kc) * rms(a) * rms(b)


# The products are returned in BF16 (the gradient dtype, transformers PR #50031
# `_dequantize_fp8_weight(..., grad_output.dtype)`), so every output element carries one
# final rounding to BF16 of at most half a unit in the last place, i.e. <= 2^-8 |value|.
# That rounding is part of the method's result, not accumulation error; the elementwise
# bound is applied on top of it.  (For long contractions it is negligible against the
# bound; for an expert with one or two rows it is the whole error.)
BF16_OUTPUT_ROUNDING = 2.0 ** -8


def check(out, ref, bound, rel_fro=5e-3, out_rounding=BF16_OUTPUT_ROUNDING):
    """Return (ok, max_abs_err, rel_frobenius) for an output against its float64 reference.

    Elementwise: |out - ref| <= bound + out_rounding * |ref|.  ``bound`` may be a scalar
    or an array broadcastable to ``out``.  A zero bound with a zero reference requires
    exact zeros (an empty contraction).
    """
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(out - ref)
    max_err = float(err.max()) if err.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(out - ref) / nref) if nref > 0 else (0.0 if max_err == 0 else np.inf)
    ok = bool(np.all(err <= bound + out_rounding * np.abs(ref))) and rel <= rel_fro and np.all(np.isfinite(out))
    return ok, max_err, rel
