"""Thin ctypes binding of libsage_gb300.so -- argument marshalling only.

Every function here has the name of the C entry point it wraps.  Device memory (outputs and the
workspace) comes from PyTorch; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: without the built library, or without a CUDA device, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsage_gb300.so")

SAGE_OK, SAGE_ERR_ARG, SAGE_ERR_UNSUPPORTED, SAGE_ERR_ALIGN = 0, 1, 2, 3
SAGE_ERR_CUDA, SAGE_ERR_TIMEOUT, SAGE_ERR_WORKSPACE = 4, 5, 6
SAGE_FP16, SAGE_BF16 = 0, 1
SAGE_FLAG_DUMP = 1
SAGE_FLAG_DP_INT8 = 2
SAGE_FLAG_FP8 = 4
SAGE_FLAG_OPS16 = 8

EXPORTED = (
    "sage_quantize_workspace_bytes", "sage_quantize_smooth", "sage_fwd_workspace_bytes",
    "sage_attn_fwd", "sage_bwd_workspace_bytes", "sage_attn_bwd", "sage_dump_bytes",
    "sage_device_status", "sage_status_string", "sage_version", "sage_quantize_smooth_qknorm",
    "sage_qknorm_bwd", "sage_quantize_fp4", "sage_attn_fwd_fp4",
)


class SageParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
        ("dtype", ctypes.c_int), ("causal", ctypes.c_int), ("smooth_k", ctypes.c_int),
        ("smooth_q", ctypes.c_int), ("flags", ctypes.c_uint), ("dump", ctypes.c_void_p),
        ("dump_bytes", ctypes.c_size_t), ("ops16", ctypes.c_void_p),
    ]


class SageQkNorm(ctypes.Structure):
    """struct sage_qknorm (include/sage.h)."""
    _fields_ = [
        ("gQ", ctypes.c_void_p), ("gK", ctypes.c_void_p), ("eps", ctypes.c_float),
        ("rQ", ctypes.c_void_p), ("rK", ctypes.c_void_p), ("Qn", ctypes.c_void_p),
        ("Kn", ctypes.c_void_p),
    ]


class SageError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m bit_trainable_attention_sage_gb300.build` "
            "(the SageBwd library has no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(SageParams)
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    for name in ("sage_quantize_workspace_bytes", "sage_fwd_workspace_bytes", "sage_bwd_workspace_bytes",
                 "sage_qat_bwd_workspace_bytes"):
        getattr(L, name).argtypes = [P]
        getattr(L, name).restype = sz
    L.sage_dump_bytes.argtypes = [P, ci]
    L.sage_dump_bytes.restype = sz
    L.sage_quantize_smooth.argtypes = [P] + [vp] * 12 + [sz, vp]
    L.sage_quantize_smooth.restype = ci
    L.sage_quantize_smooth_qknorm.argtypes = [P, ctypes.POINTER(SageQkNorm)] + [vp] * 12 + [sz, vp]
    L.sage_quantize_smooth_qknorm.restype = ci
    L.sage_qknorm_bwd.argtypes = [P] + [vp] * 6 + [vp]
    L.sage_qknorm_bwd.restype = ci
    L.sage_quantize_fp4.argtypes = [P] + [vp] * 12 + [sz, vp]
    L.sage_quantize_fp4.restype = ci
    L.sage_attn_fwd_fp4.argtypes = [P] + [vp] * 12 + [sz, vp]
    L.sage_attn_fwd_fp4.restype = ci
    L.sage_attn_fwd.argtypes = [P] + [vp] * 12 + [sz, vp]
    L.sage_attn_fwd.restype = ci
    L.sage_attn_bwd.argtypes = [P] + [vp] * 15 + [sz, vp]
    L.sage_attn_bwd.restype = ci
    L.sage_qat_quantize.argtypes = [P] + [vp] * 6 + [vp]
    L.sage_qat_quantize.restype = ci
    L.sage_qat_fwd.argtypes = [P] + [vp] * 7 + [vp]
    L.sage_qat_fwd.restype = ci
    L.sage_qat_bwd.argtypes = [P] + [vp] * 11 + [sz, vp]
    L.sage_qat_bwd.restype = ci
    L.sage_device_status.argtypes = [vp]
    L.sage_device_status.restype = ci
    L.sage_status_string.argtypes = [ci]
    L.sage_status_string.restype = ctypes.c_char_p
    L.sage_version.argtypes = []
    L.sage_version.restype = ctypes.c_char_p
    L.sage_quantize_noalloc_max_partials.argtypes = []
    L.sage_quantize_noalloc_max_partials.restype = sz
    L.sage_quantize_noalloc_partials_needed.argtypes = [P]
    L.sage_quantize_noalloc_partials_needed.restype = sz
    L.sage_quantize_smooth_noalloc.argtypes = [P] + [vp] * 12
    L.sage_quantize_smooth_noalloc.restype = ci
    _lib = L
    return L


def _check(fn: str, status: int):
    if status != SAGE_OK:
        raise SageError(fn, status, lib().sage_status_string(status).decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return SAGE_FP16
    if t.dtype == torch.bfloat16:
        return SAGE_BF16
    raise TypeError(f"SageBwd takes fp16 or bf16 tensors, got {t.dtype}")


def make_params(B: int, H: int, N: int, d: int, dtype: int, causal: bool, smooth_k: bool = True,
                smooth_q: bool = False, dump: torch.Tensor | None = None, fp8: bool = False,
                ops16: torch.Tensor | None = None) -> SageParams:
    p = SageParams(B, H, N, d, dtype, int(causal), int(smooth_k), int(smooth_q), 0, None, 0, None)
    if fp8:
        p.flags |= SAGE_FLAG_FP8
    if ops16 is not None:
        p.flags |= SAGE_FLAG_OPS16
        p.ops16 = ops16.data_ptr()
    if dump is not None:
        p.flags |= SAGE_FLAG_DUMP
        p.dump = dump.data_ptr()
        p.dump_bytes = dump.numel() * dump.element_size()
    return p


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("SageBwd tensors must be contiguous CUDA tensors")


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


@dataclass
class Quantized:
    """The quantised forward inputs (codes, scales, means) and the problem description.
    With ``fp8`` the int8 code tensors hold FP8 E4M3 bit patterns (SAGE_FLAG_FP8), and the
    forward and backward calls on this object run the FP8 variant."""
    Qh: torch.Tensor
    Kh: torch.Tensor
    Vh: torch.Tensor
    sQ: torch.Tensor
    sK: torch.Tensor
    sV: torch.Tensor
    muK: torch.Tensor
    muQ: torch.Tensor | None
    dtype: int
    smooth_k: bool
    smooth_q: bool
    fp8: bool = False
    # QK-norm prologue (sage_quantize_smooth_qknorm): row factors and, when kept, normalised Q, K
    rQ: torch.Tensor | None = None
    rK: torch.Tensor | None = None
    Qn: torch.Tensor | None = None
    Kn: torch.Tensor | None = None
    # SAGE_FLAG_OPS16: (3,B,H,N,d) fp16 values of the Q^, K^, V^ codes, read by the forward and
    # backward calls instead of widening the codes again
    ops16: torch.Tensor | None = None


def _ops16_buffer(B, H, N, d, dev, want: bool) -> torch.Tensor | None:
    return torch.empty((3, B, H, N, d), dtype=torch.float16, device=dev) if want else None


def sage_quantize_smooth(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, smooth_k: bool = True,
                         smooth_q: bool = False, fp8: bool = False, ops16: bool = True,
                         stream=None) -> Quantized:
    """K-smoothing (+ optional Q-smoothing) and per-block INT8 (``fp8``: E4M3) quantisation of
    (B,H,N,d) Q, K, V.  With ``ops16`` (the default) the call also writes the codes' fp16 values,
    which the forward and backward calls on the result then read instead of widening the codes."""
    _require_cuda(Q, K, V)
    B, H, N, d = Q.shape
    dt = _dtype_code(Q)
    dev = Q.device
    o16 = _ops16_buffer(B, H, N, d, dev, ops16)
    p = make_params(B, H, N, d, dt, False, smooth_k, smooth_q, fp8=fp8, ops16=o16)
    Qh = torch.empty((B, H, N, d), dtype=torch.int8, device=dev)
    Kh, Vh = torch.empty_like(Qh), torch.empty_like(Qh)
    sQ = torch.empty((B, H, N // 64), dtype=torch.float32, device=dev)
    sK, sV = torch.empty_like(sQ), torch.empty_like(sQ)
    muK = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    muQ = torch.empty((B, H, N // 64, d), dtype=torch.float32, device=dev) if smooth_q else None
    L = lib()
    nws = L.sage_quantize_workspace_bytes(ctypes.byref(p))
    ws = _workspace(nws, dev)
    st = L.sage_quantize_smooth(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(Qh), _ptr(Kh), _ptr(Vh),
                                _ptr(sQ), _ptr(sK), _ptr(sV), _ptr(muK), _ptr(muQ), _ptr(ws), nws,
                                _stream(stream))
    _check("sage_quantize_smooth", st)
    return Quantized(Qh, Kh, Vh, sQ, sK, sV, muK, muQ, dt, smooth_k, smooth_q, fp8, ops16=o16)


def sage_quantize_smooth_qknorm(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *,
                                gamma_q: torch.Tensor | None = None, gamma_k: torch.Tensor | None = None,
                                eps: float = 1e-6, smooth_k: bool = True, smooth_q: bool = False,
                                fp8: bool = False, keep_normed: bool = False, ops16: bool = True,
                                stream=None) -> Quantized:
    """QK-norm (per-token RMSNorm of Q and K, float32 gammas of d entries or None) fused into
    sage_quantize_smooth.  The result carries the row factors rQ, rK and, with ``keep_normed``
    (forced when ``smooth_q``), the normalised Q and K; pass ``q.Kn`` as K to the forward and
    backward calls when ``smooth_q``."""
    _require_cuda(Q, K, V, gamma_q, gamma_k)
    B, H, N, d = Q.shape
    dt = _dtype_code(Q)
    dev = Q.device
    o16 = _ops16_buffer(B, H, N, d, dev, ops16)
    p = make_params(B, H, N, d, dt, False, smooth_k, smooth_q, fp8=fp8, ops16=o16)
    Qh = torch.empty((B, H, N, d), dtype=torch.int8, device=dev)
    Kh, Vh = torch.empty_like(Qh), torch.empty_like(Qh)
    sQ = torch.empty((B, H, N // 64), dtype=torch.float32, device=dev)
    sK, sV = torch.empty_like(sQ), torch.empty_like(sQ)
    muK = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    muQ = torch.empty((B, H, N // 64, d), dtype=torch.float32, device=dev) if smooth_q else None
    rQ = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    rK = torch.empty_like(rQ)
    keep = keep_normed or smooth_q
    Qn = torch.empty_like(Q) if keep else None
    Kn = torch.empty_like(K) if keep else None
    qn = SageQkNorm(_ptr(gamma_q), _ptr(gamma_k), float(eps), _ptr(rQ), _ptr(rK), _ptr(Qn), _ptr(Kn))
    L = lib()
    nws = L.sage_quantize_workspace_bytes(ctypes.byref(p))
    ws = _workspace(nws, dev)
    st = L.sage_quantize_smooth_qknorm(ctypes.byref(p), ctypes.byref(qn), _ptr(Q), _ptr(K), _ptr(V),
                                       _ptr(Qh), _ptr(Kh), _ptr(Vh), _ptr(sQ), _ptr(sK), _ptr(sV),
                                       _ptr(muK), _ptr(muQ), _ptr(ws), nws, _stream(stream))
    _check("sage_quantize_smooth_qknorm", st)
    return Quantized(Qh, Kh, Vh, sQ, sK, sV, muK, muQ, dt, smooth_k, smooth_q, fp8, rQ, rK, Qn, Kn, ops16=o16)


def sage_qknorm_bwd(X: torch.Tensor, r: torch.Tensor, dY: torch.Tensor, *, gamma: torch.Tensor | None = None,
                    want_dgamma: bool = True, stream=None):
    """Gradient of the QK-norm for the raw tensor X (Q or K) given the row factors r of the
    forward call and dY (float32), the gradient for the normalised tensor.  Returns (dX float32,
    dgamma float32 (d) or None)."""
    _require_cuda(X, r, dY, gamma)
    B, H, N, d = X.shape
    dev = X.device
    p = make_params(B, H, N, d, _dtype_code(X), False)
    dX = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dg = torch.empty(d, dtype=torch.float32, device=dev) if want_dgamma else None
    st = lib().sage_qknorm_bwd(ctypes.byref(p), _ptr(X), _ptr(gamma), _ptr(r), _ptr(dY), _ptr(dX),
                               _ptr(dg), _stream(stream))
    _check("sage_qknorm_bwd", st)
    return dX, dg


@dataclass
class Fp4Quantized:
    """NVFP4 inputs of the FP4 inference forward: packed E2M1 codes (uint8, two a byte) and E4M3
    scale bytes -- sQ, sK (B,H,N,d/16) along d, sV (B,H,N/16,d) along the tokens -- plus means."""
    Qc: torch.Tensor
    Kc: torch.Tensor
    Vc: torch.Tensor
    sQ: torch.Tensor
    sK: torch.Tensor
    sV: torch.Tensor
    muK: torch.Tensor
    muQ: torch.Tensor | None
    dtype: int
    smooth_k: bool
    smooth_q: bool


def sage_quantize_fp4(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, smooth_k: bool = True,
                      smooth_q: bool = False, stream=None) -> Fp4Quantized:
    """Smoothing and NVFP4 quantisation (1 x 16 blocks, E4M3 scales) of (B,H,N,d) Q, K, V."""
    _require_cuda(Q, K, V)
    B, H, N, d = Q.shape
    dt = _dtype_code(Q)
    dev = Q.device
    p = make_params(B, H, N, d, dt, False, smooth_k, smooth_q)
    u8 = dict(dtype=torch.uint8, device=dev)
    Qc, Kc, Vc = (torch.empty((B, H, N, d // 2), **u8) for _ in range(3))
    sQ, sK = (torch.empty((B, H, N, d // 16), **u8) for _ in range(2))
    sV = torch.empty((B, H, N // 16, d), **u8)
    muK = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    muQ = torch.empty((B, H, N // 64, d), dtype=torch.float32, device=dev) if smooth_q else None
    L = lib()
    nws = L.sage_quantize_workspace_bytes(ctypes.byref(p))
    ws = _workspace(nws, dev)
    st = L.sage_quantize_fp4(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(Qc), _ptr(Kc), _ptr(Vc),
                             _ptr(sQ), _ptr(sK), _ptr(sV), _ptr(muK), _ptr(muQ), _ptr(ws), nws, _stream(stream))
    _check("sage_quantize_fp4", st)
    return Fp4Quantized(Qc, Kc, Vc, sQ, sK, sV, muK, muQ, dt, smooth_k, smooth_q)


def sage_attn_fwd_fp4(q: Fp4Quantized, *, causal: bool, K: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None):
    """SageAttention3 FP4 inference forward.  Returns (O in the input dtype, L float32)."""
    B, H, N, d = q.Qc.shape[0], q.Qc.shape[1], q.Qc.shape[2], 2 * q.Qc.shape[3]
    dev = q.Qc.device
    p = make_params(B, H, N, d, q.dtype, causal, q.smooth_k, q.smooth_q)
    odt = torch.float16 if q.dtype == SAGE_FP16 else torch.bfloat16
    O = torch.empty((B, H, N, d), dtype=odt, device=dev) if out is None else out
    Lse = torch.empty((B, H, N), dtype=torch.float32, device=dev) if lse is None else lse
    _require_cuda(O, Lse, K)
    L = lib()
    nws = L.sage_fwd_workspace_bytes(ctypes.byref(p))
    ws = workspace if workspace is not None else _workspace(nws, dev)
    st = L.sage_attn_fwd_fp4(ctypes.byref(p), _ptr(q.Qc), _ptr(q.Kc), _ptr(q.Vc), _ptr(q.sQ), _ptr(q.sK),
                             _ptr(q.sV), _ptr(K), _ptr(q.muK), _ptr(q.muQ), _ptr(O), _ptr(Lse), _ptr(ws),
                             nws if ws is None else ws.numel(), _stream(stream))
    _check("sage_attn_fwd_fp4", st)
    return O, Lse


def sage_attn_fwd(q: Quantized, *, causal: bool, K: torch.Tensor | None = None,
                  out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, dump: torch.Tensor | None = None,
                  stream=None):
    """SageBwd forward.  Returns (O (B,H,N,d) in the input dtype, L (B,H,N) float32)."""
    B, H, N, d = q.Qh.shape
    dev = q.Qh.device
    p = make_params(B, H, N, d, q.dtype, causal, q.smooth_k, q.smooth_q, dump, q.fp8, q.ops16)
    odt = torch.float16 if q.dtype == SAGE_FP16 else torch.bfloat16
    O = torch.empty((B, H, N, d), dtype=odt, device=dev) if out is None else out
    Lse = torch.empty((B, H, N), dtype=torch.float32, device=dev) if lse is None else lse
    _require_cuda(O, Lse, K)
    L = lib()
    nws = L.sage_fwd_workspace_bytes(ctypes.byref(p))
    ws = workspace if workspace is not None else _workspace(nws, dev)
    st = L.sage_attn_fwd(ctypes.byref(p), _ptr(q.Qh), _ptr(q.Kh), _ptr(q.Vh), _ptr(q.sQ), _ptr(q.sK),
                         _ptr(q.sV), _ptr(K), _ptr(q.muK), _ptr(q.muQ), _ptr(O), _ptr(Lse), _ptr(ws),
                         nws if ws is None else ws.numel(), _stream(stream))
    _check("sage_attn_fwd", st)
    return O, Lse


def sage_attn_bwd(q: Quantized, V: torch.Tensor, O: torch.Tensor, L: torch.Tensor, dO: torch.Tensor, *,
                  causal: bool, K: torch.Tensor | None = None, grads=None,
                  workspace: torch.Tensor | None = None, dump: torch.Tensor | None = None, stream=None,
                  dp_int8: bool = False):
    """SageBwd backward.  Returns (dQ, dK, dV), float32 (B,H,N,d).  ``dp_int8`` selects the
    INT8-dP ablation (SAGE_FLAG_DP_INT8)."""
    _require_cuda(V, O, L, dO, K)
    B, H, N, d = q.Qh.shape
    dev = q.Qh.device
    p = make_params(B, H, N, d, q.dtype, causal, q.smooth_k, q.smooth_q, dump, q.fp8, q.ops16)
    if dp_int8:
        p.flags |= SAGE_FLAG_DP_INT8
    if grads is None:
        grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for _ in range(3))
    dQ, dK, dV = grads
    lb = lib()
    nws = lb.sage_bwd_workspace_bytes(ctypes.byref(p))
    ws = workspace if workspace is not None else _workspace(nws, dev)
    st = lb.sage_attn_bwd(ctypes.byref(p), _ptr(q.Qh), _ptr(q.Kh), _ptr(q.sQ), _ptr(q.sK), _ptr(K),
                          _ptr(q.muK), _ptr(q.muQ), _ptr(V), _ptr(O), _ptr(L), _ptr(dO), _ptr(dQ),
                          _ptr(dK), _ptr(dV), _ptr(ws), nws if ws is None else ws.numel(),
                          _stream(stream))
    _check("sage_attn_bwd", st)
    return dQ, dK, dV


def _qat_params(t: torch.Tensor, causal: bool) -> SageParams:
    B, H, N, d = t.shape
    return make_params(B, H, N, d, _dtype_code(t), causal, smooth_k=False, smooth_q=False)


def sage_qat_quantize(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, out=None, stream=None):
    """Attn-QAT NVFP4 fake quantisation (no smoothing).  Returns (Qf, Kf, Vf) in the input dtype."""
    _require_cuda(Q, K, V)
    Qf, Kf, Vf = out if out is not None else (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V))
    p = _qat_params(Q, False)
    st = lib().sage_qat_quantize(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(Qf), _ptr(Kf), _ptr(Vf),
                                 _stream(stream))
    _check("sage_qat_quantize", st)
    return Qf, Kf, Vf


def sage_qat_fwd(Qf: torch.Tensor, Kf: torch.Tensor, Vf: torch.Tensor, *, causal: bool, out=None, stream=None):
    """Attn-QAT forward.  Returns (O input dtype, O' float32, L float32 (B,H,N),
    R float32 (B,H,N/64,N) the row maxima the backward needs)."""
    _require_cuda(Qf, Kf, Vf)
    B, H, N, d = Qf.shape
    dev = Qf.device
    if out is None:
        out = (torch.empty_like(Qf), torch.empty((B, H, N, d), dtype=torch.float32, device=dev),
               torch.empty((B, H, N), dtype=torch.float32, device=dev),
               torch.empty((B, H, N // 64, N), dtype=torch.float32, device=dev))
    O, Op, Lse, R = out
    _require_cuda(O, Op, Lse, R)
    p = _qat_params(Qf, causal)
    st = lib().sage_qat_fwd(ctypes.byref(p), _ptr(Qf), _ptr(Kf), _ptr(Vf), _ptr(O), _ptr(Op), _ptr(Lse), _ptr(R),
                            _stream(stream))
    _check("sage_qat_fwd", st)
    return O, Op, Lse, R


def sage_qat_bwd(Qf: torch.Tensor, Kf: torch.Tensor, Vf: torch.Tensor, Op: torch.Tensor, L: torch.Tensor,
                 R: torch.Tensor, dO: torch.Tensor, *, causal: bool, grads=None,
                 workspace: torch.Tensor | None = None, stream=None):
    """Attn-QAT backward.  Returns (dQ, dK, dV) float32 (B,H,N,d)."""
    _require_cuda(Qf, Kf, Vf, Op, L, R, dO)
    B, H, N, d = Qf.shape
    dev = Qf.device
    if grads is None:
        grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for _ in range(3))
    dQ, dK, dV = grads
    p = _qat_params(Qf, causal)
    lb = lib()
    nws = lb.sage_qat_bwd_workspace_bytes(ctypes.byref(p))
    ws = workspace if workspace is not None else _workspace(nws, dev)
    st = lb.sage_qat_bwd(ctypes.byref(p), _ptr(Qf), _ptr(Kf), _ptr(Vf), _ptr(Op), _ptr(L), _ptr(R), _ptr(dO),
                         _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), nws if ws is None else ws.numel(), _stream(stream))
    _check("sage_qat_bwd", st)
    return dQ, dK, dV


def sage_dump_bytes(B, H, N, d, which: int) -> int:
    p = make_params(B, H, N, d, SAGE_FP16, False)
    return lib().sage_dump_bytes(ctypes.byref(p), which)


def sage_device_status(stream=None) -> int:
    """Waits for the stream; SAGE_OK or SAGE_ERR_TIMEOUT (a bounded device wait expired)."""
    return lib().sage_device_status(_stream(stream))


def sage_version() -> str:
    return lib().sage_version().decode()


def sage_status_string(status: int) -> str:
    return lib().sage_status_string(status).decode()


def sage_quantize_smooth_noalloc(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *,
                                 smooth_k: bool = True, smooth_q: bool = False, fp8: bool = False,
                                 ops16: bool = True, out=None, stream=None) -> Quantized:
    """sage_quantize_smooth for callers that cannot allocate device memory while they run: the
    K-mean scratch lives in a fixed array inside the library.  ``out`` (a Quantized whose tensors
    the caller allocated beforehand) receives the results; without it they are allocated here."""
    _require_cuda(Q, K, V)
    B, H, N, d = Q.shape
    dt = _dtype_code(Q)
    dev = Q.device
    if out is None:
        Qh = torch.empty((B, H, N, d), dtype=torch.int8, device=dev)
        sQ = torch.empty((B, H, N // 64), dtype=torch.float32, device=dev)
        out = Quantized(Qh, torch.empty_like(Qh), torch.empty_like(Qh), sQ, torch.empty_like(sQ),
                        torch.empty_like(sQ), torch.empty((B, H, d), dtype=torch.float32, device=dev),
                        torch.empty((B, H, N // 64, d), dtype=torch.float32, device=dev) if smooth_q else None,
                        dt, smooth_k, smooth_q, fp8, ops16=_ops16_buffer(B, H, N, d, dev, ops16))
    L = lib()
    fn = L.sage_quantize_smooth_noalloc
    p = make_params(B, H, N, d, dt, False, smooth_k, smooth_q, fp8=fp8, ops16=out.ops16)
    st = fn(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(out.Qh), _ptr(out.Kh), _ptr(out.Vh),
            _ptr(out.sQ), _ptr(out.sK), _ptr(out.sV), _ptr(out.muK), _ptr(out.muQ), _stream(stream))
    _check("sage_quantize_smooth_noalloc", st)
    return out
