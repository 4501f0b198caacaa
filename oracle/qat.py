"""Oracle: Attn-QAT attention, forward and backward (TEST INFRASTRUCTURE, not product code).

"Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (technical summary):
  * section 2.1: the backward recomputes P, and the softmax gradient relies on
    rowsum(P o dP) = rowsum(dO o O), which holds only if the forward and the backward compute P
    in the same precision;
  * section 2.2: (i) when the backward recomputes P it applies the same FP4 fake quantisation the
    forward applied; (ii) the forward also produces a high-precision output O', and the backward
    forms the scalar term from dO and O' alone; (iii) no Q/K smoothing and no two-level P scaling;
  * section 2.3: FP4 is the NVFP4 format of "SageAttention3 ..." (review) (E2M1 values, 1 x 16
    blocks, E4M3 scales; oracle.fp4), and the backward runs in BF16 ("high precision").

Readings where the pages leave a step open (the plainest ones the rest supports):
  Q1  Q, K and V are fake-quantised once, Q' = s Q^ etc., with the NVFP4 quantiser of oracle.fp4
      (Q, K blocked along d, V along the tokens, the contraction axis of P V), no smoothing.  The
      values s * code have at most 6 significant bits and lie in [2^-10, 2688], so they are exact
      in fp16 and in bf16: every matrix product below runs on the input 16-bit type.
  Q2  forward logits and softmax follow the per-tile form of the INT8 forward: per 64-key block,
      acc = Q' K'^T (exact), c = fl32(log2(e)/sqrt(d)), the logits S_k = fl32(acc_k c) as float32
      values, r = max_k S_k over the unmasked keys, x_k = fl32(S_k - r), e_k = fl32(2^x_k); l
      accumulates the unquantised e (eq. (1) of "SageAttention3 ..." (review)), m the running max
      of r.
  Q3  phi, the P fake quantiser, is one-level NVFP4 along the keys: per 16 keys of a row,
      s = e4m3(fl32(max e / 6)), codes e2m1(fl32(e * fl32(1/s))), P^ = codes * s (a zero scale
      gives zero codes).  The forward applies it to e (each 64-key block normalised by its own
      row max r, so the block's largest entry is 1) and keeps r (float32, one per row and key
      block).  "The same quantisation as the forward" in the backward is read as rebuilding the
      forward's quantised P exactly: e = fl32(2^fl32(S - r)) from the stored r, phi(e), then
      normalised, P^ = rnd16(fl32(phi(e) * fl32(2^(fl32(r - L2))))), so that dV is the gradient of the
      forward's own O with respect to V'.  (phi of the normalised P itself would not do: in a
      diffuse row of 8192 keys P is near 1.2e-4 and max / 6 lies far below the smallest E4M3
      scale 2^-9, so whole blocks would quantise to zero.)
  Q4  O = sum_j 2^(r_j - m) P^_j V'_j / l in the input dtype; O' = sum_j 2^(r_j - m) rnd16(e_j) V'_j
      / l kept in float32: the unquantised P~ enters its product as a 16-bit operand (BF16 is the
      pages' "high precision"), exactly as the backward's products do.
  Q5  backward: P = fl32(2^(fl32(S - L2))) with L2 = fl32(L log2(e)); D = rowsum(dO o O');
      dP = fl32(dO V'^T); dS = fl32(P fl32(dP - D)) rounded to the input dtype for the two
      products it feeds; dV = P^^T dO (P^ of Q3), dQ = dS K' / sqrt(d), dK = dS^T Q' / sqrt(d)
      (the fake quantisers pass the gradient straight through, so these are also the gradients
      of Q, K and V).

Exactness: each float32 rounding the readings name is taken here (fl32 below);
products of fake-quantised operands are exact in float64 (at most 12 significant bits each, a
row of 128 sums stays exact unless its products span more than 2^34); everything that only
accumulates (m, l, O, O', D, dQ, dK, dV) is float64.  ``exact=True`` replaces every quantiser and
every rounding by the identity: the same tiled code must then equal float64 full-precision
attention and its gradients (oracle.fpa), which pins the tiling, O', D and the backward structure.

Parity: pinned by tests/test_oracle_qat.py (the identity limit against oracle.fpa, the P fake
quantiser against a brute-force grid search, a hand-worked block, the forward against its
untiled closed form, the rowsum identity behind O', dV as the exact gradient of the forward's O
with respect to V', the straight-through gradient, and the pages' ablation ordering: D from the
FP4 output O is further from the straight-through gradient than D from O').
"""
from __future__ import annotations

import math

import numpy as np

from .fp4 import dequant, e2m1_round, nvfp4_quant
from .quant import e4m3_round

F32 = np.float32
LOG2E = 1.4426950408889634
LN2 = 0.6931471805599453
BLOCK = 64


def _fl32(x, exact: bool):
    return np.asarray(x, np.float64) if exact else np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def fake_quant(Q, K, V, exact: bool = False) -> dict:
    """Q1: the fake-quantised Q', K', V' (float64 holding exact values)."""
    if exact:
        return dict(Qf=np.asarray(Q, np.float64), Kf=np.asarray(K, np.float64), Vf=np.asarray(V, np.float64))
    out = {}
    for name, x, axis in (("Qf", Q, -1), ("Kf", K, -1), ("Vf", V, -2)):
        codes, scales = nvfp4_quant(np.asarray(x, np.float32), axis=axis)
        out[name] = dequant(codes, scales, axis=axis)
    return out


def p_fake_quant(p) -> np.ndarray:
    """Q3: phi over the last axis (a multiple of 16) of float32 values p >= 0; float64 result."""
    p = np.asarray(p, np.float32)
    *lead, n = p.shape
    blocks = p.reshape(*lead, n // 16, 16)
    s = e4m3_round((blocks.max(axis=-1) / F32(6)).astype(np.float32)).astype(np.float32)
    inv = np.where(s == 0, F32(0), F32(1) / np.where(s == 0, F32(1), s)).astype(np.float32)
    codes = e2m1_round((blocks * inv[..., None]).astype(np.float32))
    return (codes * s[..., None].astype(np.float64)).reshape(*lead, n)


def _mask(causal: bool, i: int, j: int):
    if causal and i == j:
        return ~np.triu(np.ones((BLOCK, BLOCK), bool), k=1)
    return np.ones((BLOCK, BLOCK), bool)


def qat_forward(fq: dict, causal: bool, dtype_round, exact: bool = False, heads=None, q_blocks=None):
    """Q2-Q4.  Returns (O, O', L, R): O, O', L float64 (O before its rounding to the stored
    dtype), R (B, H, N/64, N) the row maxima r of each (key block, row), float32 values (-inf
    where the row sees no key of the block; NaN where the forward never visits the pair)."""
    Qf, Kf, Vf = fq["Qf"], fq["Kf"], fq["Vf"]
    B, H, N, d = Qf.shape
    T = N // BLOCK
    c = LOG2E / math.sqrt(d) if exact else float(F32(LOG2E / math.sqrt(d)))
    O = np.zeros((B, H, N, d))
    Op = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    R = np.full((B, H, T, N), np.nan)
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for (b, h) in heads:
        for i in (q_blocks if q_blocks is not None else range(T)):
            rows = slice(BLOCK * i, BLOCK * i + BLOCK)
            m = np.full(BLOCK, -np.inf)
            l = np.zeros(BLOCK)
            acc_o = np.zeros((BLOCK, d))
            acc_p = np.zeros((BLOCK, d))
            for j in range(T):
                if causal and j > i:
                    break
                cols = slice(BLOCK * j, BLOCK * j + BLOCK)
                valid = _mask(causal, i, j)
                acc = Qf[b, h, rows] @ Kf[b, h, cols].T
                S = _fl32(acc * c, exact)
                r = np.where(valid, S, -np.inf).max(axis=1)
                R[b, h, j, rows] = r
                x = np.where(valid, _fl32(S - np.where(np.isfinite(r), r, 0.0)[:, None], exact), -np.inf)
                e = _fl32(np.exp2(x), exact)
                p_hat = e if exact else p_fake_quant(e)
                p_16 = e if exact else np.asarray(dtype_round(e.astype(np.float32)), np.float64)
                m_new = np.maximum(m, r)
                alpha = np.exp2(m - m_new)
                g = np.exp2(r - m_new)
                l = alpha * l + g * e.sum(axis=1)
                acc_o = alpha[:, None] * acc_o + g[:, None] * (p_hat @ Vf[b, h, cols])
                acc_p = alpha[:, None] * acc_p + g[:, None] * (p_16 @ Vf[b, h, cols])
                m = m_new
            O[b, h, rows] = acc_o / l[:, None]
            Op[b, h, rows] = acc_p / l[:, None]
            L[b, h, rows] = (m + np.log2(l)) * LN2
    return O, Op, L, R


def qat_backward(fq: dict, Op_stored, L_stored, R, dO, causal: bool, dtype_round, exact: bool = False,
                 heads=None, q_blocks=None, kv_blocks=None, D_from=None, bwd_p_quant: bool = True):
    """Q5.  ``Op_stored``: O' as stored (float32), ``L_stored``: the stored float32 L, ``R`` the
    forward's row maxima, ``dO`` the 16-bit upstream gradient.  ``q_blocks`` / ``kv_blocks`` restrict which dQ / dK, dV rows are
    completed.  The two ablations of section 2.2 / the results: ``D_from`` replaces O' in D (D
    from the FP4 output O), ``bwd_p_quant=False`` feeds dV the unquantised P.
    Returns dict(dQ, dK, dV, D) float64."""
    Qf, Kf, Vf = fq["Qf"], fq["Kf"], fq["Vf"]
    B, H, N, d = Qf.shape
    T = N // BLOCK
    c = LOG2E / math.sqrt(d) if exact else float(F32(LOG2E / math.sqrt(d)))
    inv_sqrt_d = 1.0 / math.sqrt(d)
    dO = np.asarray(dO, np.float64)
    src = Op_stored if D_from is None else D_from
    D = (dO * np.asarray(src, np.float64)).sum(axis=-1)
    D32 = _fl32(D, exact)
    if exact:
        L2 = np.asarray(L_stored, np.float64) * LOG2E
    else:
        L2 = (np.asarray(L_stored, np.float32) * F32(LOG2E)).astype(np.float32).astype(np.float64)
    dQ = np.zeros((B, H, N, d))
    dK = np.zeros((B, H, N, d))
    dV = np.zeros((B, H, N, d))
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]

    def tile(b, h, i, j, want_dq, want_dkv):
        rows = slice(BLOCK * i, BLOCK * i + BLOCK)
        cols = slice(BLOCK * j, BLOCK * j + BLOCK)
        valid = _mask(causal, i, j)
        acc = Qf[b, h, rows] @ Kf[b, h, cols].T
        S = _fl32(acc * c, exact)
        x = np.where(valid, _fl32(S - L2[b, h, rows][:, None], exact), -np.inf)
        P = _fl32(np.exp2(x), exact)
        dP = _fl32(dO[b, h, rows] @ Vf[b, h, cols].T, exact)
        dS = _fl32(P * _fl32(dP - D32[b, h, rows][:, None], exact), exact)
        dS16 = dS if exact else np.asarray(dtype_round(dS.astype(np.float32)), np.float64)
        if want_dkv:
            if exact or not bwd_p_quant:
                p_hat = P
            else:
                # Q3: the forward's quantised P, rebuilt from its row maxima and normalised
                r = np.asarray(R[b, h, j, rows], np.float64)
                live = valid.any(axis=1)
                r0 = np.where(live, r, 0.0)
                e = np.where(valid, _fl32(np.exp2(_fl32(S - r0[:, None], False)), False), 0.0)
                g = _fl32(np.exp2(_fl32(r0 - L2[b, h, rows], False)), False)
                p_hat = np.where(live[:, None], _fl32(p_fake_quant(e) * g[:, None], False), 0.0)
                p_hat = np.asarray(dtype_round(p_hat.astype(np.float32)), np.float64)
            dV[b, h, cols] += p_hat.T @ dO[b, h, rows]
            dK[b, h, cols] += inv_sqrt_d * (dS16.T @ Qf[b, h, rows])
        if want_dq:
            dQ[b, h, rows] += inv_sqrt_d * (dS16 @ Kf[b, h, cols])

    for (b, h) in heads:
        if q_blocks is None and kv_blocks is None:
            for j in range(T):
                for i in range(j if causal else 0, T):
                    tile(b, h, i, j, True, True)
        else:
            for j in (kv_blocks or []):
                for i in range(j if causal else 0, T):
                    tile(b, h, i, j, False, True)
            for i in (q_blocks or []):
                for j in range(0, (i + 1) if causal else T):
                    tile(b, h, i, j, True, False)
    return dict(dQ=dQ, dK=dK, dV=dV, D=D)


def run(Q, K, V, dO, causal: bool, dtype_round, exact: bool = False) -> dict:
    """Whole Attn-QAT path on full tensors: fake quantisation, forward, backward."""
    fq = fake_quant(Q, K, V, exact=exact)
    O, Op, L, R = qat_forward(fq, causal, dtype_round, exact=exact)
    Op_stored = Op if exact else Op.astype(np.float32)
    L_stored = L if exact else L.astype(np.float32)
    O_stored = O if exact else dtype_round(O.astype(np.float32))
    g = qat_backward(fq, Op_stored, L_stored, R, dO, causal, dtype_round, exact=exact)
    return dict(fq=fq, O=O, Op=Op, L=L, R=R, O_stored=O_stored, Op_stored=Op_stored, L_stored=L_stored, **g)
