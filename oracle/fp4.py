"""Oracle: SageAttention3 FP4 inference forward (TEST INFRASTRUCTURE, not product code).

"SageAttention3: Microscaling FP4 Attention for Inference and An Exploration of 8-Bit Training"
(review):
  * FP4 microscaling quantisation, eq. (2)-(3): X is split into 1 x n blocks along the contraction
    dimension, s = max|X_block| / 6, X^ = FP4 rounding of X / s, X' = s X^;
  * the format table: NVFP4, E2M1 values, 1 x 16 blocks, E4M3 (FP8) scale factors;
  * eq. (4)-(5): S = FP4MM(Q^, s_Q, K^, s_K), online softmax, P^ = phi(P~), V^ = phi(V),
    O = FP4MM(P^, s_P, V^, s_V);
  * two-level P scaling, eq. (6): s_P1 = rowmax(P~) / (448 x 6), P~2 = P~ / s_P1,
    (s_P2, P^2) = phi(P~2), O = FP4MM(P^2, s_P2, V^, s_V) x s_P1;
  * with Q- and K-smoothing (the review's "smoothing Q+K" row).

Readings where the pages leave a step open:
  * E2M1 is 1 sign, 2 exponent bits (bias 1), 1 mantissa bit: values 0, 0.5, 1, 1.5, 2, 3, 4, 6;
    FP4 rounding is round to nearest, ties to the even mantissa, saturating at +-6;
  * a block scale is s = e4m3(fl32(max|x| / 6)) (the E4M3 value nearest, ties even); codes are
    e2m1(fl32(x / s)) with IEEE float32 division; a block whose scale is 0 has all-zero codes;
  * Q and K (after smoothing) are blocked along d, V along the tokens (the contraction of P V),
    16 consecutive tokens per channel;
  * the softmax follows the INT8 path's per-tile form (R7): the logits are the float32 values
    S = fl32(acc c), c = fl32(log2(e) / sqrt(d)) (the block scales live inside the dequantised
    operands), r is the row max of S over the 64-key tile and x = fl32(S - r);
    P~2 = fl32(2688 fl32(2^x)) and s_P1 = 2^(r - m) / 2688, which is eq. (6) with
    rowmax(P~) = 2^(r - m); the second level quantises P~2 in 1 x 16 blocks along the keys with
    codes e2m1(fl32(v * fl32(1 / s_P2))): the reciprocal of each block scale formed once, as the
    backward's INT8 tiles form theirs (R8);
  * l accumulates the unquantised P~ as in eq. (1); Q-smoothing adds the same bias as R5, in a
    second float32 rounding S = fl32(fl32(acc c) + b).

The block products of dequantised FP4 operands are computed in float64 (each operand has at most
6 significant bits, an E2M1 value 1.1b times an E4M3 scale 1.xxxb, so each product at most 12; a
sum of 128 of them is exact unless its products span more than 2^34 in magnitude).

Parity: pinned by tests/test_oracle_fp4.py (E2M1 rounding against the nearest point of the
decoded 16-pattern grid, a hand-worked block with scale rounding and saturation, the forward
against its order-independent closed form, FP4 less accurate than INT8).
"""
from __future__ import annotations

import math

import numpy as np

from .quant import e4m3_round, k_mean, q_block_mean

F32 = np.float32
LOG2E = 1.4426950408889634
LN2 = 0.6931471805599453
P2_MAX = 448.0 * 6.0            # 2688: the first level maps each row's P~ max here


def e2m1_round(y) -> np.ndarray:
    """Nearest E2M1 value (ties to even mantissa, saturating at +-6).  Below 2 the values are
    spaced 0.5 (0, 0.5 subnormal; 1, 1.5), in [2, 4) by 1, in [4, 8) by 2 (4 and 6 only)."""
    y = np.asarray(y, np.float64)
    a = np.abs(y)
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    q = np.minimum(np.rint(a / quantum) * quantum, 6.0)
    return np.copysign(q, y)


def e2m1_decode(nibble) -> np.ndarray:
    """Value of E2M1 bit patterns (0..15): sign bit 3, exponent bits 2-1, mantissa bit 0."""
    b = np.asarray(nibble, np.int64) & 15
    sign = np.where(b & 8, -1.0, 1.0)
    e = (b >> 1) & 3
    m = b & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.ldexp(1.0, e - 1))
    return sign * mag


def nvfp4_quant(x, axis: int = -1) -> tuple[np.ndarray, np.ndarray]:
    """phi(X): 1 x 16 blocks along ``axis``.  Returns (codes as E2M1 values (float32, same shape as
    x), scales (float32, that axis divided by 16))."""
    x = np.moveaxis(np.asarray(x, np.float32), axis, -1)
    *lead, n = x.shape
    if n % 16:
        raise ValueError("the blocked axis must be a multiple of 16")
    blocks = x.reshape(*lead, n // 16, 16)
    mx = np.abs(blocks).max(axis=-1)
    s = e4m3_round((mx / F32(6)).astype(np.float32)).astype(np.float32)     # float32 division
    safe = np.where(s == 0, F32(1), s)
    y = (blocks / safe[..., None]).astype(np.float32)                          # IEEE float32 division
    codes = np.where(s[..., None] == 0, 0.0, e2m1_round(y)).astype(np.float32)
    codes = np.moveaxis(codes.reshape(*lead, n), -1, axis)
    return codes, np.moveaxis(s, -1, axis if axis >= 0 else axis)


def dequant(codes, scales, axis: int = -1) -> np.ndarray:
    """X' = s X^ (exact: at most 6 significant bits)."""
    c = np.moveaxis(np.asarray(codes, np.float64), axis, -1)
    s = np.moveaxis(np.asarray(scales, np.float64), axis, -1)
    return np.moveaxis(c * np.repeat(s, 16, axis=-1), -1, axis)


def quantize_fp4(Q, K, V, smooth_k: bool = True, smooth_q: bool = False) -> dict:
    """Smoothing as in the INT8 path (oracle.quant), then phi of Q, K along d and of V along N."""
    Q = np.asarray(Q, np.float32)
    K = np.asarray(K, np.float32)
    V = np.asarray(V, np.float32)
    B, H, N, d = K.shape
    muK = k_mean(K) if smooth_k else np.zeros((B, H, d), np.float32)
    Ksm = (K - muK[:, :, None, :]).astype(np.float32)
    muQ = None
    Qsm = Q
    if smooth_q:
        muQ = q_block_mean(Q)
        Qsm = (Q.reshape(B, H, N // 64, 64, d) - muQ[:, :, :, None, :]).reshape(B, H, N, d).astype(np.float32)
    Qc, sQ = nvfp4_quant(Qsm, axis=-1)
    Kc, sK = nvfp4_quant(Ksm, axis=-1)
    Vc, sV = nvfp4_quant(V, axis=-2)
    return dict(Qc=Qc, sQ=sQ, Kc=Kc, sK=sK, Vc=Vc, sV=sV, muK=muK, muQ=muQ, Ksm=Ksm)


def p_two_level(x) -> tuple[np.ndarray, np.ndarray]:
    """Second level of eq. (6) on one tile of logits x (rows x keys, keys a multiple of 16):
    v = fl32(2688 fl32(2^x)); per 16 keys s2 = e4m3(fl32(max v / 6)), codes e2m1(fl32(v fl32(1/s2))).
    Returns (2^x in float64, the dequantised P' = codes s2 (float64))."""
    e64 = np.exp2(np.asarray(x, np.float32).astype(np.float64))
    v = (F32(P2_MAX) * e64.astype(np.float32)).astype(np.float32)
    rows, n = v.shape
    vb = v.reshape(rows, n // 16, 16)
    s2 = e4m3_round((vb.max(axis=-1) / F32(6)).astype(np.float32)).astype(np.float32)
    inv = np.where(s2 == 0, F32(0), F32(1) / np.where(s2 == 0, F32(1), s2)).astype(np.float32)
    codes = e2m1_round((vb * inv[..., None]).astype(np.float32))
    return e64, (codes * s2[..., None].astype(np.float64)).reshape(rows, n)


def sage_fp4_forward(prep: dict, causal: bool, heads=None):
    """SageAttention3 FP4 forward over 64 x 64 tiles.  Returns (O float64, L float64)."""
    Qd = dequant(prep["Qc"], prep["sQ"], axis=-1)
    Kd = dequant(prep["Kc"], prep["sK"], axis=-1)
    Vd = dequant(prep["Vc"], prep["sV"], axis=-2)
    B, H, N, d = Qd.shape
    T = N // 64
    c = float(F32(LOG2E / math.sqrt(d)))
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    tri = np.triu(np.ones((64, 64), bool), k=1)
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for (b, h) in heads:
        for i in range(T):
            rows = slice(64 * i, 64 * i + 64)
            m = np.full(64, -np.inf)
            l = np.zeros(64)
            acc = np.zeros((64, d))
            bias = None
            if prep.get("muQ") is not None:
                mu = np.asarray(prep["muQ"][b, h, i], np.float64)
                bias = (np.asarray(prep["Ksm"][b, h], np.float64) @ mu).astype(np.float32) * F32(c)
            for j in range(T):
                if causal and j > i:
                    break
                cols = slice(64 * j, 64 * j + 64)
                s = Qd[b, h, rows] @ Kd[b, h, cols].T
                valid = ~tri if (causal and j == i) else np.ones((64, 64), bool)
                # the logits as float32 values S = fl32(acc c) (+ bias: fl32(S + b)), x = fl32(S - r)
                S = (s * c).astype(np.float32)
                if bias is not None:
                    S = (S + bias[cols][None, :]).astype(np.float32)
                r = np.where(valid, S, -np.inf).max(axis=1).astype(np.float32)
                x = (S - np.where(np.isfinite(r), r, F32(0))[:, None]).astype(np.float32)
                x = np.where(valid, x, -np.inf)
                e64, pd = p_two_level(x)
                m_new = np.maximum(m, r.astype(np.float64))
                alpha = np.exp2(m - m_new)
                g = np.exp2(r.astype(np.float64) - m_new)
                l = alpha * l + g * e64.sum(axis=1)
                acc = alpha[:, None] * acc + (g / P2_MAX)[:, None] * (pd @ Vd[b, h, cols])
                m = m_new
            O[b, h, rows] = acc / l[:, None]
            L[b, h, rows] = (m + np.log2(l)) * LN2
    return O, L
