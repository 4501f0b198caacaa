"""Oracle: per-block INT8 (or FP8 E4M3) quantisation and smoothing (TEST INFRASTRUCTURE, not
product code).

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

FP8 variant ("SageAttention3 ..." (review), "INT8 vs FP8 training": the same SageBwd with FP8
instead of INT8 codes).  The pages give only the comparison; the plainest reading keeps every
step and swaps the code format: E4M3 of the OCP 8-bit floating-point format (1 sign, 4 exponent
bits with bias 7, 3 mantissa bits; subnormals k 2^-9; largest finite 448; no infinities),
delta = fl32(max|x| / 448), code = e4m3_round(fl32(x / delta)): round to the nearest E4M3 value,
ties to the even mantissa, magnitudes beyond 448 saturating to 448.

Parity: pinned by tests/test_oracle_quant.py (hand-worked block, exact-rational re-derivation
over every finite fp16 value, zero block, mean exactness) and tests/test_oracle_fp8.py (E4M3
rounding against the nearest point of the decoded 256-pattern grid, hand-worked ties and
saturation).
"""
from __future__ import annotations

import numpy as np

BLOCK = 64
F32 = np.float32
E4M3_MAX = 448.0
QMAX = {"int8": 127, "e4m3": 448}


def e4m3_round(y) -> np.ndarray:
    """Round float values to the nearest finite E4M3 value (ties to even mantissa, saturating).

    Binade [2^e, 2^(e+1)) with e >= -6 holds 8 values 2^e (1 + m/8), a quantum of 2^(e-3); below
    2^-6 the subnormals k 2^-9 share the quantum 2^-9.  Dividing by a power of two is exact, so
    rint (ties to even) on the scaled value rounds once, and an even rint result is an even
    mantissa -- carries into the next binade land on its (even) leading value.
    """
    y = np.asarray(y, np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)                         # a = f 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = np.maximum(ex - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    q = np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX)
    return np.copysign(q, y)


def e4m3_decode(byte) -> np.ndarray:
    """Value of E4M3 bit patterns (uint8): sign bit 7, exponent bits 6-3, mantissa bits 2-0.
    The two NaN patterns (exponent and mantissa all ones) decode to NaN."""
    b = np.asarray(byte, np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.ldexp(1.0, e - 10))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(v) -> np.ndarray:
    """Bit pattern (uint8) of values that are E4M3 values (the inverse of e4m3_decode); -0 keeps
    its sign bit."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0)
    _, ex = np.frexp(a)
    e = ex - 1                                  # floor(log2 a) for a > 0
    normal = a >= 2.0 ** -6
    ebits = np.where(normal, e + 7, 0)
    mbits = np.where(normal, np.rint(np.ldexp(a, -np.where(normal, e, 0) + 3)) - 8, np.rint(a * 2.0 ** 9))
    out = (sign | (ebits.astype(np.int64) << 3) | mbits.astype(np.int64)).astype(np.uint8)
    assert np.array_equal(e4m3_decode(out), np.where(np.signbit(v), -a, a)), "not an E4M3 value"
    return out


def quantize_block(x, fmt: str = "int8") -> tuple[np.ndarray, np.float32]:
    """Quantise one block (any shape) of float32 values; returns (codes, float32 delta).

    fmt "int8": int8 codes; fmt "e4m3": the E4M3 code values as float32 (exact)."""
    x = np.asarray(x, dtype=np.float32)
    ctype = np.int8 if fmt == "int8" else np.float32
    if x.size == 0:
        return np.zeros(x.shape, ctype), F32(0)
    mx = np.max(np.abs(x))
    delta = F32(mx) / F32(QMAX[fmt])
    if delta == 0:
        return np.zeros(x.shape, ctype), F32(0)
    y = x / delta                          # float32 / float32 is IEEE round-to-nearest
    if fmt == "e4m3":
        return e4m3_round(y).astype(np.float32), F32(delta)
    q = np.clip(np.rint(y), -127, 127).astype(np.int8)    # rint ties to even
    return q, F32(delta)


def quantize_per_block(x, block: int = BLOCK, fmt: str = "int8") -> tuple[np.ndarray, np.ndarray]:
    """Quantise (..., N, d) float32 values in blocks of ``block`` tokens x d.

    Returns codes (..., N, d) (int8, or E4M3 values as float32) and float32 scales
    (..., N / block).  Each block goes through :func:`quantize_block` one at a time.
    """
    x = np.asarray(x, dtype=np.float32)
    *lead, n, d = x.shape
    if n % block:
        raise ValueError("N must be a multiple of the block size")
    flat = x.reshape(-1, n // block, block, d)
    codes = np.empty(flat.shape, np.int8 if fmt == "int8" else np.float32)
    scales = np.empty(flat.shape[:2], np.float32)
    for h in range(flat.shape[0]):
        for b in range(flat.shape[1]):
            codes[h, b], scales[h, b] = quantize_block(flat[h, b], fmt)
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


def quantize_smooth(Q, K, V, smooth_k: bool = True, smooth_q: bool = False, fmt: str = "int8") -> dict:
    """Steps a1 + a2: K-mean, optional Q-block-mean, smoothing and per-block quantisation.

    Inputs are float32 arrays (B, H, N, d) holding the 16-bit input values exactly.
    Returns dict(Qh, Kh, Vh codes (int8, or E4M3 values as float32 for fmt "e4m3"); sQ, sK, sV
    float32 (B, H, N/64); muK (B, H, d) float32 or zeros; muQ (B, H, N/64, d) float32 or None;
    Ksm float32 (B, H, N, d) -- the smoothed K, kept only for the Q-smoothing bias term).
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
    Qh, sQ = quantize_per_block(Qsm, fmt=fmt)
    Kh, sK = quantize_per_block(Ksm, fmt=fmt)
    Vh, sV = quantize_per_block(V, fmt=fmt)
    return dict(Qh=Qh, Kh=Kh, Vh=Vh, sQ=sQ, sK=sK, sV=sV, muK=muK, muQ=muQ, Ksm=Ksm)
