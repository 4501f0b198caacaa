"""Oracle: float64 full-precision attention (FPA) and its gradients (TEST INFRASTRUCTURE).

Scaled dot-product attention as defined on "SageBwd: A Trainable Low-bit Attention" (section
summary, 3 Preliminaries: S = QK^T, P = softmax(S), O = PV) with the 1/sqrt(d) of the QK-norm
paragraph of the structured summary, and its gradients from the structured summary's
"attention gradients" paragraph: dV = P^T dO, dP = dO V^T, dS = P o (dP - delta) with
delta = rowsum(dO o O), dQ = dS K, dK = dS^T Q (each of the last two times 1/sqrt(d)).

Plain dense float64 matrices; the causal mask is top-left aligned (key <= query).
Parity: pinned by central finite differences and the identities in tests/test_oracle_fpa.py.
"""
from __future__ import annotations

import math

import numpy as np


def _scores(Q, K, causal):
    d = Q.shape[-1]
    S = np.asarray(Q, np.float64) @ np.swapaxes(np.asarray(K, np.float64), -1, -2) / math.sqrt(d)
    if causal:
        n = S.shape[-1]
        S = np.where(np.triu(np.ones((n, n), bool), k=1), -np.inf, S)
    return S


def softmax_rows(S):
    M = S.max(axis=-1, keepdims=True)
    E = np.exp(S - M)
    return E / E.sum(axis=-1, keepdims=True)


def fpa_forward(Q, K, V, causal: bool = False):
    """Returns (O, L, P): output, natural-log LSE of the scaled scores, and the softmax."""
    S = _scores(Q, K, causal)
    M = S.max(axis=-1, keepdims=True)
    E = np.exp(S - M)
    lsum = E.sum(axis=-1, keepdims=True)
    P = E / lsum
    O = P @ np.asarray(V, np.float64)
    L = (M + np.log(lsum))[..., 0]
    return O, L, P


def fpa_backward(Q, K, V, dO, causal: bool = False, O=None):
    """Returns dict(dQ, dK, dV, P, dP, dS, D).  ``O`` defaults to the float64 forward output."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    d = Q.shape[-1]
    O_f, _, P = fpa_forward(Q, K, V, causal)
    O = O_f if O is None else np.asarray(O, np.float64)
    dV = np.swapaxes(P, -1, -2) @ dO
    dP = dO @ np.swapaxes(V, -1, -2)
    D = (dO * O).sum(axis=-1)
    dS = P * (dP - D[..., None])
    dQ = dS @ K / math.sqrt(d)
    dK = np.swapaxes(dS, -1, -2) @ Q / math.sqrt(d)
    return dict(dQ=dQ, dK=dK, dV=dV, P=P, dP=dP, dS=dS, D=D)
