"""Oracle: per-block INT8 quantisation and smoothing (TEST INFRASTRUCTURE, not product code).

Follows:
  * "SageBwd: A Trainable Low-bit Attention" (structured summary), prerequisites, "INT8
    quantisation": X^ = round(X / delta_X), delta_X = max|X| / 127, per-block granularity
    aligned with the FlashAttention tiles.
  * "SageAttention3: Microscaling FP4 Attention for Inference and An Exploration of 8-Bit
    Training" (review), eq. (7): s_X = max|X| / 127 per block.
  * "SageBwd: A Trainable Low-bit Attention" (structured summary), prerequisites, "K-smoothing
    and Q-smoothing": mu_K = mean over tokens of K, K_sm = K - mu_K; mu_Qi = mean over the rows
    of query block i, Q_sm = Q - mu_Qi.

Readings where the pages leave a step open (each is a documented constant of the contract):
  * the block is 64 tokens x the full head dimension, for Q, K, V and dO;
  * delta = fl32(max|x| / 127); q = clamp(round_half_even(fl32(x / delta)), -127, 127) with
    IEEE float32 division -- the pages only say "round";
  * a block whose max is zero (or whose delta underflows to zero) gets delta = 0 and q = 0;
  * mu_K is the float64 sum over all N tokens divided by N in float64, rounded once to float32,
    whether or not the attention is causal; mu_Q is the same over the 64 rows of each block;
  * the smoothed value fl32(x - mu) is quantised directly and never stored.

Parity: pinned by tests/test_oracle_quant.py (hand-worked block, exact-rational re-derivation
over every finite fp16 value, zero block, mean exactness).
"""
from __future__ import annotations

import numpy as np

BLOCK = 64
F32 = np.float32


def quantize_block(x) -> tuple[np.ndarray, np.float32]:
    """Quantise one block (any shape) of float32 values; returns (int8 codes, float32 delta)."""
    x = np.asarray(x, dtype=np.float32)
    if x.size == 0:
        return np.zeros(x.shape, np.int8), F32(0)
    mx = np.max(np.abs(x))
    delta = F32(mx) / F32(127)
    if delta == 0:
        return np.zeros(x.shape, np.int8), F32(0)
    q = np.rint(x / delta)                # float32 / float32 is IEEE round-to-nearest; rint ties to even
    q = np.clip(q, -127, 127).astype(np.int8)
    return q, F32(delta)


def quantize_per_block(x, block: int = BLOCK) -> tuple[np.ndarray, np.ndarray]:
    """Quantise (..., N, d) float32 values in blocks of ``block`` tokens x d.

    Returns int8 codes (..., N, d) and float32 scales (..., N / block).  Each block goes through
    :func:`quantize_block` one at a time.
    """
    x = np.asarray(x, dtype=np.float32)
    *lead, n, d = x.shape
    if n % block:
        raise ValueError("N must be a multiple of the block size")
    flat = x.reshape(-1, n // block, block, d)
    codes = np.empty(flat.shape, np.int8)
    scales = np.empty(flat.shape[:2], np.float32)
    for h in range(flat.shape[0]):
        for b in range(flat.shape[1]):
            codes[h, b], scales[h, b] = quantize_block(flat[h, b])
    return codes.reshape(x.shape), scales.reshape(*lead, n // block)


def k_mean(k) -> np.ndarray:
    """mu_K[..., c] = (1/N) sum_n K[..., n, c]: float64 sum, float64 divide, one float32 rounding."""
    k64 = np.asarray(k, dtype=np.float64)
    n = k64.shape[-2]
    return (k64.sum(axis=-2) / n).astype(np.float32)


def q_block_mean(q, block: int = BLOCK) -> np.ndarray:
    """mu_Q[..., i, c] = mean over the ``block`` rows of query block i (same rounding as k_mean)."""
    q64 = np.asarray(q, dtype=np.float64)
    *lead, n, d = q64.shape
    blocks = q64.reshape(*lead, n // block, block, d)
    return (blocks.sum(axis=-2) / block).astype(np.float32)


def quantize_smooth(Q, K, V, smooth_k: bool = True, smooth_q: bool = False) -> dict:
    """Steps a1 + a2: K-mean, optional Q-block-mean, smoothing and per-block quantisation.

    Inputs are float32 arrays (B, H, N, d) holding the 16-bit input values exactly.
    Returns dict(Qh, Kh, Vh int8; sQ, sK, sV float32 (B, H, N/64); muK (B, H, d) float32 or
    zeros; muQ (B, H, N/64, d) float32 or None; Ksm float32 (B, H, N, d) -- the smoothed K,
    kept only for the Q-smoothing bias term).
    """
    Q = np.asarray(Q, np.float32)
    K = np.asarray(K, np.float32)
    V = np.asarray(V, np.float32)
    B, H, N, d = K.shape
    muK = k_mean(K) if smooth_k else np.zeros((B, H, d), np.float32)
    Ksm = (K - muK[:, :, None, :]).astype(np.float32)          # float32 subtraction, one rounding
    if smooth_q:
        muQ = q_block_mean(Q)
        Qsm = (Q.reshape(B, H, N // BLOCK, BLOCK, d) - muQ[:, :, :, None, :]).reshape(B, H, N, d)
        Qsm = Qsm.astype(np.float32)
    else:
        muQ = None
        Qsm = Q
    Qh, sQ = quantize_per_block(Qsm)
    Kh, sK = quantize_per_block(Ksm)
    Vh, sV = quantize_per_block(V)
    return dict(Qh=Qh, Kh=Kh, Vh=Vh, sQ=sQ, sK=sK, sV=sV, muK=muK, muQ=muQ, Ksm=Ksm)
