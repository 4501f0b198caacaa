"""SageBwd as a differentiable PyTorch operation.

``sage_attention(Q, K, V, causal=...)`` runs the quantise + forward calls of the C library and
records what the backward call needs; ``.backward()`` runs ``sage_attn_bwd``.  Every step runs in
the library's kernels: this module only keeps tensors alive between the two calls and converts
the float32 gradients to the inputs' dtype.

K-smoothing needs no backward term: K_sm = K - 1 mu_K^T, and the correction -(1/N) 1 (1^T dK_sm)
vanishes because the rows of dS sum to zero ("SageBwd: A Trainable Low-bit Attention", section
summary, K-smoothing).  With Q-smoothing the library adds the dK bias term itself.
"""
import torch

from .binding import sage_attn_bwd, sage_attn_fwd, sage_quantize_smooth


class SageAttentionFunction(torch.autograd.Function):
    """O = SageBwd attention(Q, K, V); inputs (B, H, N, d) fp16 or bf16 CUDA tensors."""

    @staticmethod
    def forward(ctx, Q, K, V, causal: bool, smooth_q: bool, dp_int8: bool, fp8: bool):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        q = sage_quantize_smooth(Q, K, V, smooth_q=smooth_q, fp8=fp8)
        O, L = sage_attn_fwd(q, causal=causal, K=K if smooth_q else None)
        ctx.q = q
        ctx.causal, ctx.smooth_q, ctx.dp_int8 = causal, smooth_q, dp_int8
        ctx.save_for_backward(K, V, O, L)
        return O

    @staticmethod
    def backward(ctx, dO):
        K, V, O, L = ctx.saved_tensors
        q = ctx.q
        dQ, dK, dV = sage_attn_bwd(q, V, O, L, dO.to(O.dtype).contiguous(), causal=ctx.causal,
                                   K=K if ctx.smooth_q else None, dp_int8=ctx.dp_int8)
        del ctx.q
        return dQ.to(O.dtype), dK.to(O.dtype), dV.to(O.dtype), None, None, None, None


def sage_attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False,
                   smooth_q: bool = False, dp_int8: bool = False, fp8: bool = False) -> torch.Tensor:
    """Differentiable SageBwd attention (softmax(Q K^T / sqrt(d)) V with INT8 quantisation;
    ``fp8`` selects the FP8 E4M3 variant, ``dp_int8`` the INT8-dP ablation)."""
    return SageAttentionFunction.apply(Q, K, V, causal, smooth_q, dp_int8, fp8)
