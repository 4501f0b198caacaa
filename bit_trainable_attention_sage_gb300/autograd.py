"""SageBwd as a differentiable PyTorch operation.

``sage_attention(Q, K, V, causal=...)`` runs the quantise + forward calls of the C library and
records what the backward call needs; ``.backward()`` runs ``sage_attn_bwd``.  Every step runs in
the library's kernels: this module only keeps tensors alive between the calls and converts the
float32 gradients to the inputs' dtypes.

K-smoothing needs no backward term: K_sm = K - 1 mu_K^T, and the correction -(1/N) 1 (1^T dK_sm)
vanishes because the rows of dS sum to zero ("SageBwd: A Trainable Low-bit Attention", section
summary, K-smoothing).  With Q-smoothing the library adds the dK bias term itself.

With ``qk_norm`` the quantiser first RMS-normalises Q and K per token ("SageBwd ..." (structured
summary), QK-norm: x / sqrt(mean x^2 + eps) * gamma) and the backward chains the attention
gradients through ``sage_qknorm_bwd``, which also gives the gradients of the two gammas.

``sage_attention_qat`` is Attn-QAT ("Attn-QAT: 4-Bit Attention With Quantization-Aware Training",
technical summary, section 2.2): the forward runs on NVFP4 fake-quantised Q, K, V with an FP4 P
and keeps the high-precision output O'; the backward rebuilds the forward's quantised P and forms
D from O'.  Fake quantisation passes the gradient straight through.
"""
import torch

from .binding import (sage_attn_bwd, sage_attn_fwd, sage_qat_bwd, sage_qat_fwd, sage_qat_quantize,
                      sage_qknorm_bwd, sage_quantize_smooth, sage_quantize_smooth_qknorm)


class SageAttentionFunction(torch.autograd.Function):
    """O = SageBwd attention(Q, K, V); inputs (B, H, N, d) fp16 or bf16 CUDA tensors, optional
    QK-norm gammas of d entries."""

    @staticmethod
    def forward(ctx, Q, K, V, gamma_q, gamma_k, causal: bool, smooth_q: bool, dp_int8: bool,
                fp8: bool, qk_norm: bool, eps: float):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        gq = gamma_q.detach().float().contiguous() if gamma_q is not None else None
        gk = gamma_k.detach().float().contiguous() if gamma_k is not None else None
        if qk_norm:
            q = sage_quantize_smooth_qknorm(Q, K, V, gamma_q=gq, gamma_k=gk, eps=eps,
                                            smooth_q=smooth_q, fp8=fp8)
            Kb = q.Kn if smooth_q else None
        else:
            q = sage_quantize_smooth(Q, K, V, smooth_q=smooth_q, fp8=fp8)
            Kb = K if smooth_q else None
        O, L = sage_attn_fwd(q, causal=causal, K=Kb)
        ctx.q, ctx.Kb, ctx.gq, ctx.gk = q, Kb, gq, gk
        ctx.causal, ctx.dp_int8, ctx.qk_norm = causal, dp_int8, qk_norm
        ctx.gdtypes = (None if gamma_q is None else gamma_q.dtype, None if gamma_k is None else gamma_k.dtype)
        ctx.save_for_backward(Q, K, V, O, L)
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, L = ctx.saved_tensors
        q = ctx.q
        dQ, dK, dV = sage_attn_bwd(q, V, O, L, dO.to(O.dtype).contiguous(), causal=ctx.causal,
                                   K=ctx.Kb, dp_int8=ctx.dp_int8)
        dgq = dgk = None
        if ctx.qk_norm:
            dQ, dgq = sage_qknorm_bwd(Q, q.rQ, dQ, gamma=ctx.gq,
                                      want_dgamma=ctx.gq is not None and ctx.needs_input_grad[3])
            dK, dgk = sage_qknorm_bwd(K, q.rK, dK, gamma=ctx.gk,
                                      want_dgamma=ctx.gk is not None and ctx.needs_input_grad[4])
            dgq = None if dgq is None else dgq.to(ctx.gdtypes[0])
            dgk = None if dgk is None else dgk.to(ctx.gdtypes[1])
        del ctx.q, ctx.Kb
        return (dQ.to(O.dtype), dK.to(O.dtype), dV.to(O.dtype), dgq, dgk,
                None, None, None, None, None, None)


def sage_attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False,
                   smooth_q: bool = False, dp_int8: bool = False, fp8: bool = False,
                   qk_norm: bool = False, gamma_q: torch.Tensor | None = None,
                   gamma_k: torch.Tensor | None = None, eps: float = 1e-6) -> torch.Tensor:
    """Differentiable SageBwd attention (softmax(Q K^T / sqrt(d)) V with INT8 quantisation;
    ``fp8`` selects the FP8 E4M3 variant, ``dp_int8`` the INT8-dP ablation, ``qk_norm`` the fused
    QK-norm prologue with optional learnable gammas)."""
    if (gamma_q is not None or gamma_k is not None) and not qk_norm:
        raise ValueError("gamma_q / gamma_k need qk_norm=True")
    return SageAttentionFunction.apply(Q, K, V, gamma_q, gamma_k, causal, smooth_q, dp_int8, fp8,
                                       qk_norm, eps)


class SageQatAttentionFunction(torch.autograd.Function):
    """O = Attn-QAT attention(Q, K, V); inputs (B, H, N, d) fp16 or bf16 CUDA tensors."""

    @staticmethod
    def forward(ctx, Q, K, V, causal: bool):
        Qf, Kf, Vf = sage_qat_quantize(Q.contiguous(), K.contiguous(), V.contiguous())
        O, Op, L, R = sage_qat_fwd(Qf, Kf, Vf, causal=causal)
        ctx.causal = causal
        ctx.save_for_backward(Qf, Kf, Vf, Op, L, R)
        return O

    @staticmethod
    def backward(ctx, dO):
        Qf, Kf, Vf, Op, L, R = ctx.saved_tensors
        dQ, dK, dV = sage_qat_bwd(Qf, Kf, Vf, Op, L, R, dO.to(Qf.dtype).contiguous(), causal=ctx.causal)
        return dQ.to(Qf.dtype), dK.to(Qf.dtype), dV.to(Qf.dtype), None


def sage_attention_qat(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False) -> torch.Tensor:
    """Differentiable Attn-QAT attention: 4-bit (NVFP4) fake-quantised forward, 16-bit backward."""
    return SageQatAttentionFunction.apply(Q, K, V, causal)
