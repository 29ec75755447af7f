"""Reference oracle for the block-scaled backward path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow CPU restatement of what the CUDA library computes:

  * decode of the packed codes (E4M3, E2M1, E8M0) by table, built from the OCP
    8-bit floating point and OCP Microscaling (MX) v1.0 definitions;
  * application of the block scales with the BF16 rounding rule
    (value cast to BF16, scale cast to BF16, product rounded to nearest even);
  * float64 matrix products for grad_X = grad_out @ W and grad_W = grad_out^T @ X,
    per expert over int32 cumulative offsets in the grouped case.

Sources (web pages on block-scaled low-precision backward passes):
  * MSLK PR #393 "Add Autograd Backward Support for FP4 GEMM Custom Ops",
    section "Implementation Method" (dequantize packed FP4 to BF16, then the two
    standard matmul gradients);
  * transformers PR #50031 "Train adapters on top of FP8 weights",
    `_dequantize_fp8_weight`, `FP8LinearFunction.backward`,
    `FP8GroupedMatmulFunction.backward` (block-scale broadcast and the grouped
    product over offsets);
  * AstrAI `astrai/extension/fp8.py`, the FP8_MAX table (E4M3 max 448).

Who may use it: only the test-suite, the package's smoke check and the CPU
baseline leg of the benchmark.  The library (``block_scaled_gemm_fp8_gb300``)
never imports this package and this package imports nothing from it; the two
share no code, tables or helpers.  Every function here is pinned by tests in
``tests/test_oracle_*.py`` against facts that do not come from the oracle
itself (library conversions, exact rational arithmetic, closed forms).
"""

from . import formats, dequant, gemm  # noqa: F401
