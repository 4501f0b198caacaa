"""SageBwd trainable INT8 attention for GB300 (sm_103a).

The compute path is the C-ABI library libsage_gb300.so (include/sage.h); this package holds its
CUDA sources (csrc/), the in-tree build (build.py) and a thin ctypes binding (binding.py) whose
functions carry the C entry points' names.  ``autograd.sage_attention`` wraps the calls as a
differentiable PyTorch operation; ``autograd.sage_attention_qat`` does the same for the Attn-QAT
calls (4-bit fake-quantised forward with a high-precision O', 16-bit backward).
"""
from .binding import (  # noqa: F401
    Fp4Quantized, Quantized, SageError, SageParams, lib, make_params, sage_attn_bwd, sage_attn_fwd,
    sage_attn_fwd_fp4, sage_quantize_fp4, sage_qat_bwd, sage_qat_fwd, sage_qat_quantize,
    sage_device_status, sage_dump_bytes, sage_qknorm_bwd, sage_quantize_smooth,
    sage_quantize_smooth_noalloc, sage_quantize_smooth_qknorm, sage_status_string, sage_version,
)
from .autograd import (SageAttentionFunction, SageQatAttentionFunction, sage_attention,  # noqa: F401,E402
                       sage_attention_qat)
