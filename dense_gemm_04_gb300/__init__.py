"""phx: a single-GPU GEMM library for GB300 (sm_103a).

C = alpha * A @ B + beta * C on row-major f32 matrices, in two precisions:

* ``sgemm``: f32 on CUDA cores (register-blocked FFMA micro-tiles, multi-stage cp.async
  shared-memory pipeline, fused alpha/beta epilogue);
* ``gemm_f16tc_f32acc``: f32 operands rounded to f16 (to nearest, ties to even), products
  summed in f32 on the tensor cores (TMA-fed swizzled stages, tcgen05.mma into TMEM).

The work happens in ``libphx.so`` behind the C ABI declared in ``include/phx.h``; the
module :mod:`dense_gemm_04_gb300.phx` is a thin ctypes binding over it.  Importing this
package does not load the CUDA library; :mod:`dense_gemm_04_gb300.phx` does, and raises if
it was not built.
"""
__all__ = ["phx", "synth"]
