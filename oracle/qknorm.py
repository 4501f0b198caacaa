"""Oracle: QK-norm (per-token RMSNorm of Q and K) and its gradient (TEST INFRASTRUCTURE, not
product code).

"SageBwd: A Trainable Low-bit Attention" (structured summary), "QK-norm": each token's query and
key vector is RMS-normalised, RMSNorm(x) = x / sqrt((1/d) sum_i x_i^2) * gamma with a learnable
scale vector gamma; reproduction paragraph: norm epsilon 1e-6 (read as added to the mean square).

Readings where the pages leave a step open:
  * r = 1 / sqrt(ms + eps) is the float32 nearest to its exact value, ms = (1/d) sum_c x_c^2 the
    exact mean square of the 16-bit inputs and eps the float32 value the caller passes (1e-6 in
    the pages' setup): computed here as the exact sum of squares rounded once to float64
    (math.fsum), divided by d (a power of two, exact), then IEEE float64 steps and one final
    rounding to float32, which is correctly rounded unless the exact value lies within about
    2^-52 of a float32 rounding boundary;
  * the normalised value is y = round_dtype(fl32(fl32(x * r) * gamma_c)): the fused prologue
    produces exactly what a separate norm writing a 16-bit tensor would, and everything after it
    (K-mean, smoothing, quantisation) runs on those 16-bit values;
  * gamma has d entries shared by every head and token (NULL / None = ones);
  * the backward treats the final rounding to 16 bits as the identity and differentiates
    y = gamma * x * r in float64: dx = r (gamma * dy - xh * mean_c(gamma_c dy_c xh_c)),
    xh = x * r; dgamma_c = sum over all tokens of dy_c xh_c.

Parity: pinned by tests/test_oracle_qknorm.py (r against the exact value by bracketing its
float32 neighbours' midpoints in rational arithmetic, central finite differences of the float64
function, the gradient's orthogonality to x at eps = 0, bit-exact invariance under power-of-two
scaling, a hand-worked row).
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32


def row_factor(x, eps: float) -> np.ndarray:
    """r = fl32(1 / sqrt(fl64(fsum(x^2)) / d + eps)) per row of (..., d) 16-bit values."""
    x = np.asarray(x, np.float32).astype(np.float64)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    ss = np.array([math.fsum(v * v for v in row) for row in flat])    # exact sum, one rounding
    ms = ss / d
    r = 1.0 / np.sqrt(ms + float(F32(eps)))
    return r.astype(np.float32).reshape(x.shape[:-1])


def rms_norm(x, gamma, eps: float, dtype_round) -> tuple[np.ndarray, np.ndarray]:
    """Forward QK-norm of (..., d) 16-bit values held as float32.
    Returns (y: the normalised values rounded by ``dtype_round``, r float32 (...))."""
    x = np.asarray(x, np.float32)
    r = row_factor(x, eps)
    y = x * r[..., None]                                   # float32 product, one rounding
    if gamma is not None:
        y = y * np.asarray(gamma, np.float32)              # float32 product, one rounding
    return dtype_round(y.astype(np.float32)), r


def rms_norm_bwd(x, gamma, r, dy) -> tuple[np.ndarray, np.ndarray]:
    """Gradient of y = gamma * x * r(x) in float64: (dx (..., d), dgamma (d,))."""
    x = np.asarray(x, np.float64)
    r = np.asarray(r, np.float64)[..., None]
    dy = np.asarray(dy, np.float64)
    d = x.shape[-1]
    g = np.ones(d) if gamma is None else np.asarray(gamma, np.float64)
    xh = x * r
    gdy = g * dy
    dx = r * (gdy - xh * (gdy * xh).sum(axis=-1, keepdims=True) / d)
    dg = (dy * xh).reshape(-1, d).sum(axis=0)
    return dx, dg
