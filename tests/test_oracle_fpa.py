"""Pins for the float64 full-precision attention (FPA) and the metrics (CPU only).

Checks come from calculus and the pages' identities, not from the FPA itself:
  * central finite differences of the loss sum(O o dO) (attention gradients paragraph of
    "SageBwd: A Trainable Low-bit Attention", structured summary);
  * delta = rowsum(dO o O) equals rowsum(P o dP) (same paragraph);
  * softmax invariance to row constants and K - 1 mu^T (K-/Q-smoothing paragraph; section
    summary, 6 Ablation: dS rows sum to zero);
  * RMS(dS) <= max_i ||dP_i - delta_i 1||_inf / sqrt(N) (section summary, B dS magnitude).
"""
import math

import numpy as np
import pytest

from oracle import fpa, metrics


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(causal):
    N, d, h = 8, 4, 1e-6
    Q, K, V, dO = (_rand((N, d), s) for s in range(4))
    g = fpa.fpa_backward(Q, K, V, dO, causal)

    def loss(Q_, K_, V_):
        return float((fpa.fpa_forward(Q_, K_, V_, causal)[0] * dO).sum())

    for name, X, G in (("Q", Q, g["dQ"]), ("K", K, g["dK"]), ("V", V, g["dV"])):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert metrics.rel_l2(G, fd) < 1e-7, name


def test_output_is_convex_combination_and_lse():
    Q, K, V = (_rand((2, 16, 8), s) for s in range(3))
    O, L, P = fpa.fpa_forward(Q, K, V, causal=True)
    assert np.allclose(P.sum(-1), 1.0, atol=1e-14)
    assert np.all(np.triu(P[0], 1) == 0)
    S = Q @ np.swapaxes(K, -1, -2) / math.sqrt(8)
    S = np.where(np.triu(np.ones((16, 16), bool), 1), -np.inf, S)
    assert np.allclose(L, np.log(np.exp(S).sum(-1)), rtol=1e-13)
    # causal row 0 sees only key 0
    assert np.allclose(O[:, 0], V[:, 0], rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_delta_identity(causal):
    Q, K, V, dO = (_rand((3, 32, 16), s) for s in range(4))
    g = fpa.fpa_backward(Q, K, V, dO, causal)
    assert np.allclose(g["D"], (g["P"] * g["dP"]).sum(-1), rtol=1e-12, atol=1e-14)
    # hence every dS row sums to zero
    assert np.abs(g["dS"].sum(-1)).max() < 1e-12 * np.abs(g["dS"]).max() * 32


def test_smoothing_and_row_constant_invariance():
    Q, K, V, dO = (_rand((2, 32, 16), s) for s in range(4))
    K = K + 3.0
    base = fpa.fpa_forward(Q, K, V)[0]
    gb = fpa.fpa_backward(Q, K, V, dO)
    Ksm = K - K.mean(axis=-2, keepdims=True)
    assert metrics.rel_l2(fpa.fpa_forward(Q, Ksm, V)[0], base) < 1e-12
    gs = fpa.fpa_backward(Q, Ksm, V, dO)
    for k in ("dQ", "dK", "dV"):
        assert metrics.rel_l2(gs[k], gb[k]) < 1e-12, k
    # a row constant c_i added to the scores (an extra channel: c_i sqrt(17) in Q, 1 in K)
    # leaves the softmax alone
    c = _rand((2, 32, 1), 9)
    Qx = np.concatenate([Q, c * math.sqrt(17)], -1)
    Kx = np.concatenate([K, np.ones((2, 32, 1))], -1)
    Px = fpa.fpa_forward(Qx, Kx, V)[2]      # scores QK^T/sqrt(17) + c_i
    S_plain = Q @ np.swapaxes(K, -1, -2) / math.sqrt(17)
    P_plain = fpa.softmax_rows(S_plain)
    assert np.allclose(Px, P_plain, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("seed,scale,causal", [(0, 1.0, False), (1, 3.0, True), (2, 0.1, False)])
def test_ds_magnitude_bound(seed, scale, causal):
    N = 64
    Q, K, V = (_rand((1, N, 16), seed * 10 + s, scale) for s in range(3))
    dO = _rand((1, N, 16), seed * 10 + 3, 1e-2)
    g = fpa.fpa_backward(Q, K, V, dO, causal)
    rms = math.sqrt(np.mean(g["dS"] ** 2))
    bound = np.abs(g["dP"] - g["D"][..., None]).max(axis=-1).max() / math.sqrt(N)
    assert rms <= bound


def test_metrics():
    x = np.array([1.0, 2.0, 3.0])
    assert metrics.cos_sim(x, 2 * x) == pytest.approx(1.0)
    assert metrics.cos_sim([1.0, 0.0], [0.0, 1.0]) == 0.0
    assert metrics.cos_sim(x, -x) == pytest.approx(-1.0)
    assert metrics.rel_l2(1.1 * x, x) == pytest.approx(0.1)
    assert metrics.rmse([0.0, 0.0], [3.0, 4.0]) == pytest.approx(math.sqrt(12.5))
