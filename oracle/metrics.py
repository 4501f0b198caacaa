"""Oracle: error metrics (TEST INFRASTRUCTURE).

Cosine similarity sum(x y) / sqrt(sum x^2 sum y^2), relative l2 error ||x - y|| / ||y||, and the
L1 / RMSE of "SageAttention3 ..." (review), quantisation-error metric table.  All in float64.
Parity: pinned by tests/test_oracle_fpa.py (orthogonal, parallel and scaled vectors).
"""
from __future__ import annotations

import numpy as np


def cos_sim(x, y) -> float:
    x = np.asarray(x, np.float64).ravel()
    y = np.asarray(y, np.float64).ravel()
    den = np.sqrt(np.dot(x, x) * np.dot(y, y))
    return float(np.dot(x, y) / den) if den > 0 else float(np.array_equal(x, y))


def rel_l2(x, ref) -> float:
    x = np.asarray(x, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return float(num / den) if den > 0 else float(num)


def l1(x, ref) -> float:
    x = np.asarray(x, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    return float(np.abs(x - ref).sum() / max(np.abs(ref).sum(), 1e-300))


def rmse(x, ref) -> float:
    x = np.asarray(x, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    return float(np.sqrt(np.mean((x - ref) ** 2)))
