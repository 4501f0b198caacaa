"""Code-level parity of the GPU path against the oracle: where the two may differ, and by how much.

Both sides decide the P and dS codes in float32, but not by the same operations.  The oracle
takes the method's steps one correctly rounded operation at a time:
  S = fl32(acc c), x = fl32(S - r) (forward) or fl32(S - L2) (backward), P = fl32(2^x).
The kernels instead form acc c - r with one fused multiply-add and take 2^x from the hardware
approximation (relative error below 2^-21).  Their backward rounds the exact product x * (1/s)
to an integer, where the oracle rounds fl32(x * (1/s)).  Their backward also starts from the
forward's own L and D, which carry float32 accumulation errors of their own.

So a GPU code may differ from the oracle's, but only where the oracle's unrounded value y lies
within the propagated error tau of a rounding boundary: |code_gpu - y| <= 1/2 + tau.  (Usually the
codes are one apart at a half-integer; where a tile's scale itself moved, a large code can move
by more.)  Each check below bounds |y_gpu - y_oracle| from those sources, multiplies the bound by
a safety factor of 2, and asserts that every differing code lies within it.  A genuinely wrong
code does not have y near a rounding boundary and fails.  The rate of such flips is reported and
bounded separately.
"""
from __future__ import annotations

import numpy as np

LN2 = 0.6931471805599453
LOG2E32 = np.float32(1.4426950408889634)
U = 2.0 ** -24          # unit roundoff of float32
EX2 = 2.0 ** -21        # relative error bound of the hardware 2^x approximation
SAFETY = 2.0


def check_flips(gpu_codes, ref_codes, ref_y, tau, live, what):
    """Every live GPU code equals the oracle's, or is a rounding of a value within tau of the
    oracle's unrounded y: |code - y| <= 1/2 + tau.  Returns (flips, live count, the largest
    |code - y| - 1/2 over the flips: how far past the rounding boundary the GPU's value lay)."""
    g = np.asarray(gpu_codes, np.int64)[live]
    r = np.asarray(ref_codes, np.int64)[live]
    y = np.asarray(ref_y, np.float64)[live]
    t = np.asarray(tau, np.float64)[live] if np.ndim(tau) else np.full(y.shape, float(tau))
    f = g != r
    dist = np.abs(g[f] - y[f]) - 0.5
    bad = dist > t[f]
    assert not bad.any(), (what, "code away from a rounding boundary", y[f][bad][:5], g[f][bad][:5],
                           r[f][bad][:5], t[f][bad][:5])
    return int(f.sum()), int(live.sum()), float(dist.max(initial=0.0))


def fwd_code_tau(S, y, tile_r, acc_c):
    """Forward P codes: x = fl32(S - r) on the oracle side, the fused form on the GPU side.
    |dx| <= u (|acc c| + |S| + 2 |x|) (the oracle's extra rounding of acc c, a Q-smoothing bias's
    rounding, and the two sides' rounding of x); 2^x moves by ln2 |dx| plus the approximation and
    two float32 roundings; y = 127 2^x scales it."""
    S = np.asarray(S, np.float64)
    x = np.abs(S - np.asarray(tile_r, np.float64))
    eps = LN2 * U * (np.abs(acc_c) + np.abs(S) + 2 * x) + EX2 + 3 * U
    return SAFETY * np.asarray(y, np.float64) * eps + 2.0 ** -20


def l2_of(L):
    """L2 = fl32(L * fl32(log2 e)) as both sides form it from their own float32 L."""
    return (np.asarray(L, np.float32) * LOG2E32).astype(np.float32).astype(np.float64)


def bwd_tile_taus(S, acc_c, L2_ref, L2_gpu, P, dP, D_ref, D_gpu, absdp, y_p, y_ds, d, valid):
    """Bounds on |y_gpu - y_oracle| for one 64 x 64 backward tile (rows = queries).

    P: x = S - L2 moves by |dL2| (the two sides' L) plus the roundings of acc c, the bias and x
    (u (|acc c| + |S| + 2 |x|)); 2^x by ln2 |dx|
    plus the approximation.  The tile scale s = max / 127 moves with the largest relative change
    over the tile (plus the roundings of s and 1/s).  dS = P (dP - D): dP differs by the tensor
    core's float32 accumulation order (at most (d + 2) u sum |dO||V|), D by the two sides' own D,
    P as above.  Rounding the exact product x * inv instead of fl32(x * inv) adds u |y|."""
    S = np.asarray(S, np.float64)
    L2r = np.asarray(L2_ref, np.float64)[:, None]
    dL2 = np.abs(np.asarray(L2_gpu, np.float64) - np.asarray(L2_ref, np.float64))[:, None]
    x = np.abs(S - L2r)
    eps_p = LN2 * (dL2 + U * (np.abs(acc_c) + np.abs(S) + 2 * x)) + EX2 + U
    eps_p = np.where(valid, eps_p, 0.0)
    P = np.asarray(P, np.float64)
    eps_sp = eps_p.max(initial=0.0) + 2 * U
    tau_p = SAFETY * (np.abs(y_p) * (eps_p + eps_sp + 2 * U)) + 2.0 ** -20
    dPmD = np.abs(np.asarray(dP, np.float64) - np.asarray(D_ref, np.float64)[:, None])
    dD = np.abs(np.asarray(D_gpu, np.float64) - np.asarray(D_ref, np.float64))[:, None]
    d_dpmd = (d + 2) * U * np.asarray(absdp, np.float64) + dD + 2 * U * dPmD
    d_ds = P * d_dpmd + dPmD * P * eps_p + 2 * U * P * dPmD
    d_ds = np.where(valid, d_ds, 0.0)
    ds_max = (P * dPmD * valid).max(initial=0.0)
    eps_sds = (d_ds.max(initial=0.0) / ds_max if ds_max > 0 else 0.0) + 2 * U
    inv = 127.0 / ds_max if ds_max > 0 else 0.0
    tau_ds = SAFETY * (d_ds * inv + np.abs(y_ds) * (eps_sds + 2 * U)) + 2.0 ** -20
    return tau_p, tau_ds, eps_sp, eps_sds


def block_rel_l2(a, ref, block=64):
    """The largest rel-l2 error over the 64-row blocks of each head of (B, H, N, d) tensors
    (blocks whose reference is zero compare by absolute norm)."""
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    B, H, N, d = ref.shape
    worst = 0.0
    for i in range(0, N, block):
        num = np.linalg.norm((a - ref)[:, :, i:i + block].reshape(B * H, -1), axis=1)
        den = np.linalg.norm(ref[:, :, i:i + block].reshape(B * H, -1), axis=1)
        worst = max(worst, float(np.max(np.where(den > 0, num / np.where(den > 0, den, 1.0), num))))
    return worst
