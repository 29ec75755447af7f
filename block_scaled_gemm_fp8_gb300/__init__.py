"""Block-scaled low-precision backward GEMMs (dgrad / wgrad, dense and grouped) for GB300.

The compute lives in ``libbsq.so`` (hand-written sm_103a CUDA kernels behind a C ABI,
declared in ``include/bsq.h``).  ``block_scaled_gemm_fp8_gb300.bsq`` is the thin ctypes
binding with the same entry-point names; the library is loaded on first call, so that
importing this package (for example to draw synthetic inputs with
``block_scaled_gemm_fp8_gb300.synth``) needs no GPU.
"""
