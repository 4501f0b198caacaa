"""Oracle: QK-norm (per-token RMSNorm of Q and K) and its gradient (TEST INFRASTRUCTURE, not
product code).

"SageBwd: A Trainable Low-bit Attention" (structured summary), "QK-norm": each token's query and
key vector is RMS-normalised, RMSNorm(x) = x / sqrt((1/d) sum_i x_i^2) * gamma with a learnable
scale vector gamma; reproduction paragraph: norm epsilon 1e-6 (read as added to the mean square).

Readings where the pages leave a step open:
  * the sum of squares is the exact sum rounded once to float32, S = fl32(sum_c x_c^2); then, in
    IEEE float32 operations, ms = S / d (exact, d a power of two), v = fl32(ms + eps),
    s = fl32(sqrt(v)), r = fl32(1 / s); eps is a float32 value (1e-6 rounded to float32 in the
    pages' setup).  Every step is a correctly rounded float32 operation on a uniquely defined
    value, so the result does not depend on any summation order;
  * the normalised value is y = round_dtype(fl32(fl32(x * r) * gamma_c)): the fused prologue
    produces exactly what a separate norm writing a 16-bit tensor would, and everything after it
    (K-mean, smoothing, quantisation) runs on those 16-bit values;
  * gamma has d entries shared by every head and token (NULL / None = ones);
  * the backward treats the final rounding to 16 bits as the identity and differentiates
    y = gamma * x * r in float64: dx = r (gamma * dy - xh * mean_c(gamma_c dy_c xh_c)),
    xh = x * r; dgamma_c = sum over all tokens of dy_c xh_c.

Parity: pinned by tests/test_oracle_qknorm.py (central finite differences of the float64
function, the gradient's orthogonality to x at eps = 0, bit-exact invariance under power-of-two
scaling, a hand-worked row).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

F32 = np.float32


def round_f32(q: Fraction) -> np.float32:
    """The float32 nearest to a non-negative rational (ties to even); normal range only."""
    if q == 0:
        return F32(0)
    e = q.numerator.bit_length() - q.denominator.bit_length()     # 2^e <= q < 2^(e+2)
    if Fraction(2) ** e > q:
        e -= 1
    if Fraction(2) ** (e + 1) <= q:
        e += 1
    scaled = q / Fraction(2) ** (e - 23)                             # in [2^23, 2^24)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return F32(n * 2.0 ** (e - 23))


def row_factor(x, eps: float) -> np.ndarray:
    """r = fl32(1 / fl32(sqrt(fl32(fl32(sum x^2) / d + eps)))) per row of (..., d) 16-bit values,
    the sum exact before its one rounding."""
    x = np.asarray(x, np.float32)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    S = np.array([round_f32(sum(Fraction(float(v)) ** 2 for v in row)) for row in flat], np.float32)
    ms = S / F32(d)
    v = ms + F32(eps)
    r = F32(1) / np.sqrt(v)
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
