"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import workloads
from oracle import sage as osage

TORCH_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    """float32 values that are exact in ``dtype`` -> contiguous CUDA tensor of that dtype."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(TORCH_DT[dtype]).cuda()


def carve(buf: torch.Tensor, specs):
    """Split a dump buffer into consecutive 256-byte-aligned typed regions (the library's layout)."""
    out, off = [], 0
    for dtype, count in specs:
        off = (off + 255) & ~255
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        out.append(buf[off:off + nbytes].view(dtype))
        off += nbytes
    return out


def fwd_dump_views(buf, B, H, N, d):
    nn = B * H * N * N
    nb = B * H * (N // 64)
    s, p, pv = carve(buf, [(torch.int32, nn), (torch.int16, nn), (torch.int32, nb * (N // 64) * 64 * d)])
    return (s.view(B, H, N, N), p.view(B, H, N, N), pv.view(B, H, N // 64, N // 64, 64, d))


def bwd_dump_views(buf, B, H, N, d):
    nn = B * H * N * N
    nb = B * H * (N // 64)
    T = N // 64
    prod = nb * T * 64 * d
    s, p, ds, sp, sds, doh, sdo, D, dp, dv, dq, dk = carve(buf, [
        (torch.int32, nn), (torch.int16, nn), (torch.int16, nn), (torch.float32, nb * T),
        (torch.float32, nb * T), (torch.int8, B * H * N * d), (torch.float32, nb),
        (torch.float32, B * H * N), (torch.float32, nn), (torch.int32, prod), (torch.int32, prod),
        (torch.int32, prod)])
    return dict(S=s.view(B, H, N, N), P=p.view(B, H, N, N), dS=ds.view(B, H, N, N),
                sP=sp.view(B, H, T, T), sdS=sds.view(B, H, T, T),
                dOh=doh.view(B, H, N, d), sdO=sdo.view(B, H, N // 64), D=D.view(B, H, N),
                dP=dp.view(B, H, N, N), dV_int=dv.view(B, H, T, T, 64, d),
                dQ_int=dq.view(B, H, T, T, 64, d), dK_int=dk.view(B, H, T, T, 64, d))


def make_case(N, d, dtype, causal, B=1, H=2, seed=0, qk="normal", sigma=1.0, k_offset_var=0.0,
              do_var=1e-2, smooth_q=False, special=None):
    """A seeded case; ``special`` reshapes the draws into one of the method's degenerate inputs:
      "const_k"    every key of a head equal (K-smoothing makes K_sm = 0: zero K blocks, s_K = 0)
      "zero_do"    dO = 0 (every dS tile zero)
      "tiny_ds"    bf16 dO scaled per 64-row block by 2^-110, 2^-117, 2^-121, 2^-126, ... so that
                   dS tile maxima fall on both sides of the 2^-120 zero-tile bound
      "tiny_qkv"   bf16 Q and V scaled per 64-row block by 1, 2^-100, 2^-125, 2^-131, ... and K by
                   2^-127: block scales max / 127 that are subnormal in float32 (and subnormal
                   inputs)"""
    w = workloads.Workload("case", B, H, N, d, dtype, causal, qk=qk, sigma=sigma,
                           k_offset_var=k_offset_var, do_var=do_var, smooth_q=smooth_q)
    x = workloads.make_inputs(w, seed=seed)
    if special == "const_k":
        x["K"] = np.ascontiguousarray(np.broadcast_to(x["K"][:, :, :1, :], x["K"].shape))
    elif special == "zero_do":
        x["dO"] = np.zeros_like(x["dO"])
    elif special == "tiny_ds":
        assert dtype == "bf16", "the 2^-120 range needs the bf16 exponent range"
        exps = [-110, -117, -121, -126]
        per_tok = np.repeat([2.0 ** exps[i % len(exps)] for i in range(N // 64)], 64)
        x["dO"] = workloads.round_bf16((x["dO"].astype(np.float64) * per_tok[None, None, :, None]).astype(np.float32))
    elif special == "tiny_qkv":
        assert dtype == "bf16", "subnormal block scales need the bf16 exponent range"
        exps = [0, -100, -125, -131]
        per_tok = np.repeat([2.0 ** exps[i % len(exps)] for i in range(N // 64)], 64)[None, None, :, None]
        for k in ("Q", "V"):
            x[k] = workloads.round_bf16((x[k].astype(np.float64) * per_tok).astype(np.float32))
        x["K"] = workloads.round_bf16((x["K"].astype(np.float64) * 2.0 ** -127).astype(np.float32))
    elif special is not None:
        raise ValueError(special)
    return w, x


def oracle_run(w, x, record=True, dp_int8=False, fp8=False, products=False):
    rec = {} if record else None
    out = osage.run(x["Q"], x["K"], x["V"], x["dO"], w.causal,
                    lambda a: workloads.round_to(a, w.dtype), smooth_q=w.smooth_q, record=rec,
                    dp_int8=dp_int8, arith=osage.QUANTISED_FP8 if fp8 else osage.QUANTISED,
                    products=products)
    out["record"] = rec
    return out


def visited_blocks(N, causal):
    """(i, j) 64-blocks the method computes: all, or j <= i when causal."""
    T = N // 64
    return [(i, j) for i in range(T) for j in range(T) if not causal or j <= i]


def causal_mask_full(N):
    return np.triu(np.ones((N, N), bool), 1)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def oracle_fwd(w, x, record=True):
    prep = osage.prepare(x["Q"], x["K"], x["V"], smooth_q=w.smooth_q)
    rec = {} if record else None
    O, L = osage.sage_forward(prep, w.causal, record=rec)
    return prep, O, L, rec


def gpu_fwd(w, x, dump=False):
    import bit_trainable_attention_sage_gb300 as sg
    Q, K, V = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V"))
    q = sg.sage_quantize_smooth(Q, K, V, smooth_q=w.smooth_q)
    buf = None
    if dump:
        nbytes = sg.sage_dump_bytes(w.B, w.H, w.N, w.d, 0)
        buf = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    O, L = sg.sage_attn_fwd(q, causal=w.causal, K=K if w.smooth_q else None, dump=buf)
    assert sg.sage_device_status() == 0
    return dict(q=q, O=O, L=L, dump=buf, dev=dict(Q=Q, K=K, V=V))


def gpu_run(w, x, dump=False, dp_int8=False, fp8=False):
    """quantise -> forward -> backward on the GPU; returns numpy results (+ backward dump views,
    + the quantiser's outputs when fp8)."""
    import bit_trainable_attention_sage_gb300 as sg
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    q = sg.sage_quantize_smooth(Q, K, V, smooth_q=w.smooth_q, fp8=fp8)
    Kb = K if w.smooth_q else None
    O, L = sg.sage_attn_fwd(q, causal=w.causal, K=Kb)
    buf = None
    if dump:
        nbytes = sg.sage_dump_bytes(w.B, w.H, w.N, w.d, 1)
        buf = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    dQ, dK, dV = sg.sage_attn_bwd(q, V, O, L, dO, causal=w.causal, K=Kb, dump=buf, dp_int8=dp_int8)
    st = sg.sage_device_status()
    assert st == 0, sg.sage_status_string(st)
    out = dict(O=O.float().cpu().numpy(), L=L.cpu().numpy(), dQ=dQ.cpu().numpy(),
               dK=dK.cpu().numpy(), dV=dV.cpu().numpy())
    if dump:
        out["dump"] = {k: v.cpu().numpy() for k, v in bwd_dump_views(buf, w.B, w.H, w.N, w.d).items()}
    if fp8:
        out["q"] = {k: getattr(q, k).cpu().numpy() for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK")}
    return out
