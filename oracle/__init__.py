"""CPU oracle for SageBwd attention -- TEST INFRASTRUCTURE, not part of the product.

A plain, slow, obviously correct restatement of the method on the SageBwd pages, in numpy:
explicit 64-token block quantisation (float32 quantiser, round-half-even), exact integer block
products, and float64 softmax, accumulation and gradients.  It shares no code with the CUDA
library.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it; the library itself never calls into it.

Modules
  quant    per-block INT8 (and FP8 E4M3) quantiser, K-mean / Q-block-mean     (steps a1, a2, a7)
  qknorm   QK-norm (per-token RMSNorm of Q and K) and its gradient           (the prologue)
  sage     SageBwd forward (tiled online softmax, per-token P) and backward   (steps a3-a13)
  fp4      SageAttention3 FP4 (NVFP4) inference forward with two-level P scaling
  qat      Attn-QAT: NVFP4 fake-quantised forward with a high-precision O', 16-bit backward
  fpa      float64 full-precision attention and its gradients (the FPA baseline)
  metrics  cosine similarity and relative l2 error

Parity status: every function here is pinned by a ``-m "not gpu"`` test against something other
than itself (hand-worked values, exact rational re-derivation, finite differences, closed forms,
invariants).  One reported quantity is "parity unpinned": the exact Table-1 numbers of the pages'
random-QKV sweep (their N, d and block sizes are not printed), which is checked for its trend only.
"""
from . import quant, qknorm, sage, fp4, qat, fpa, metrics  # noqa: F401
from .quant import quantize_block, quantize_per_block, k_mean, quantize_smooth  # noqa: F401
from .sage import sage_forward, sage_backward, Arith, QUANTISED, QUANTISED_FP8, DEQUANTISED  # noqa: F401
from .fpa import fpa_forward, fpa_backward  # noqa: F401
