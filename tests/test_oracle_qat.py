"""Pins of the oracle's Attn-QAT path ("Attn-QAT: 4-Bit Attention With Quantization-Aware
Training", technical summary, sections 2.1-2.3), independent of the oracle's own code: float64
full-precision attention in the identity limit, a brute-force grid search for the P fake
quantiser, hand-worked blocks, untiled closed forms, the rowsum identity that O' exists for, the
straight-through gradient, and the pages' ablation ordering."""
from __future__ import annotations

import math
from fractions import Fraction as Fr

import numpy as np
import pytest

import workloads
from oracle import fp4, fpa, metrics, qat, quant
from tests.exact import fl32

E2M1_VALS = fp4.e2m1_decode(np.arange(8))
E4M3_VALS = quant.e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def _nearest(y, vals):
    """Nearest point of a sorted non-negative grid, ties to the even index (the even mantissa of
    both grids), beyond the grid its last point."""
    y = np.asarray(y, np.float64).ravel()
    dist = np.abs(y[:, None] - vals[None, :])
    tie = dist == dist.min(axis=1, keepdims=True)
    score = np.where(tie, 2 - (np.arange(len(vals))[None, :] % 2 == 0), 9)
    return vals[np.argmin(score, axis=1)]


def _phi_brute(p):
    """One-level NVFP4 of a row of non-negative float32 values, 16 at a time, by grid search and
    exact rationals: s = nearest E4M3 to fl32(max / 6), codes = nearest E2M1 to fl32(p fl32(1/s))."""
    p = np.asarray(p, np.float32).ravel()
    out = np.zeros(p.size)
    for b0 in range(0, p.size, 16):
        blk = p[b0:b0 + 16]
        mx = max(Fr(float(v)) for v in blk)
        s = float(_nearest([float(fl32(mx / 6))], E4M3_VALS)[0])
        if s == 0:
            continue
        inv = fl32(1 / Fr(s))
        y = [float(fl32(Fr(float(v)) * inv)) for v in blk]
        out[b0:b0 + 16] = _nearest(y, E2M1_VALS) * s
    return out


def _inputs(N, d, seed, dtype="fp16", causal=False):
    rng = np.random.default_rng(seed)
    Q, K, V, dO = (rng.standard_normal((1, 2, N, d)).astype(np.float32) * s for s in (1.5, 1.5, 1.0, 0.01))
    r = lambda a: workloads.round_to(a, dtype)
    return r(Q), r(K), r(V), r(dO)


@pytest.mark.parametrize("causal", [False, True])
def test_identity_limit_is_full_precision_attention(causal):
    """With every quantiser and rounding the identity, the tiled forward (O and O'), L and the
    backward equal float64 attention and its gradients."""
    Q, K, V, dO = _inputs(192, 64, seed=1, causal=causal)
    out = qat.run(Q, K, V, dO, causal, lambda a: a, exact=True)
    O_ref, L_ref, _ = fpa.fpa_forward(Q, K, V, causal)
    g = fpa.fpa_backward(Q, K, V, dO, causal)
    assert metrics.rel_l2(out["O"], O_ref) < 1e-12
    assert metrics.rel_l2(out["Op"], O_ref) < 1e-12
    assert np.max(np.abs(out["L"] - L_ref)) < 1e-12
    for k in ("dQ", "dK", "dV"):
        assert metrics.rel_l2(out[k], g[k]) < 1e-10, k


def test_p_fake_quant_hand_worked():
    """max 1: 1/6 -> E4M3 0.171875 (spacing 2^-6 in [0.125, 0.25)); 1 * fl32(1/0.171875) = 5.82 -> 6,
    0.3 -> 1.745 -> 1.5 (below the midpoint 1.75), 0.05 -> 0.29 -> 0.5.  max 0.02: 0.00333 -> the
    subnormal 2 * 2^-9; 0.02 * 256 = 5.12 -> 6.  max 1e-4: the scale rounds to 0, a zero block."""
    row = np.zeros(48, np.float32)
    row[:3] = [1.0, 0.3, 0.05]
    row[16] = 0.02
    row[32] = 1e-4
    out = qat.p_fake_quant(row[None, :])[0]
    assert out[:3].tolist() == [1.03125, 0.2578125, 0.0859375]
    assert out[16] == 6 * 2.0 ** -8 and not out[17:32].any()
    assert not out[32:].any()


def test_p_fake_quant_against_brute_force():
    rng = np.random.default_rng(5)
    rows = []
    for scale in (1.0, 0.3, 1e-2, 1e-3, 2e-4):
        rows.append((rng.random(64) * scale).astype(np.float32))
    spiky = np.exp2(-rng.uniform(0, 30, 64)).astype(np.float32)
    rows.append(spiky)
    P = np.stack(rows)
    got = qat.p_fake_quant(P)
    for r in range(P.shape[0]):
        assert np.array_equal(got[r], _phi_brute(P[r])), r


def _closed_form_forward(fq, N, d, causal, dtype):
    """Untiled: for each row and 64-key block j, the float32 logits S = fl32(acc c), r_j = max S,
    e = fl32(2^fl32(S - r_j));
    O = sum_j 2^(r_j - M) phi(e_j) V'_j / sum_j 2^(r_j - M) sum e_j, phi by grid search;
    O' the same with rnd16(e_j)."""
    Qf, Kf, Vf = (fq[k][0, 0] for k in ("Qf", "Kf", "Vf"))
    T = N // 64
    c = float(np.float32(qat.LOG2E / math.sqrt(d)))
    O = np.zeros((N, d))
    Op = np.zeros((N, d))
    for i in range(N):
        rs, ph, p16, sums, blocks = [], [], [], [], []
        for j in range(T):
            keys = np.arange(64 * j, 64 * j + 64)
            valid = keys <= i if causal else np.ones(64, bool)
            if not valid.any():
                continue
            acc = Kf[keys] @ Qf[i]
            r = float(np.float32(np.where(valid, acc, -np.inf).max() * c))
            S = (acc * c).astype(np.float32)
            x = np.where(valid, (S - np.float32(r)).astype(np.float32), -np.inf)
            e = np.exp2(x.astype(np.float64)).astype(np.float32)
            rs.append(r)
            ph.append(_phi_brute(e))
            p16.append(workloads.round_to(e, dtype).astype(np.float64))
            sums.append(e.astype(np.float64).sum())
            blocks.append(keys)
        M = max(rs)
        w = [2.0 ** (r - M) for r in rs]
        den = sum(wi * s for wi, s in zip(w, sums))
        O[i] = sum(wi * (p @ Vf[k]) for wi, p, k in zip(w, ph, blocks)) / den
        Op[i] = sum(wi * (p @ Vf[k]) for wi, p, k in zip(w, p16, blocks)) / den
    return O, Op


@pytest.mark.parametrize("causal,dtype", [(False, "fp16"), (True, "bf16")])
def test_forward_closed_form(causal, dtype):
    N, d = 128, 64
    Q, K, V, _ = _inputs(N, d, seed=3, dtype=dtype)
    fq = qat.fake_quant(Q[:, :1], K[:, :1], V[:, :1])
    O, Op, _, _ = qat.qat_forward(fq, causal, lambda a: workloads.round_to(a, dtype))
    O_cf, Op_cf = _closed_form_forward(fq, N, d, causal, dtype)
    assert metrics.rel_l2(O[0, 0], O_cf) < 1e-12
    assert metrics.rel_l2(Op[0, 0], Op_cf) < 1e-12


def test_fake_quant_values_are_exact_16bit_and_straight_through_inputs():
    """Q' etc. are the NVFP4 dequantised values: exact in fp16 and bf16, V blocked along tokens."""
    Q, K, V, _ = _inputs(64, 64, seed=4)
    fq = qat.fake_quant(Q, K, V)
    for k in ("Qf", "Kf", "Vf"):
        x = fq[k].astype(np.float32)
        assert np.array_equal(workloads.round_fp16(x), x) and np.array_equal(workloads.round_bf16(x), x), k
    codes, s = fp4.nvfp4_quant(V, axis=-2)
    assert np.array_equal(fq["Vf"], codes.astype(np.float64) * np.repeat(s, 16, axis=-2))


def test_rowsum_identity_behind_o_prime():
    """Section 2.1: rowsum(P o dP) = rowsum(dO o O') when O' carries the unquantised P.  With the
    16-bit rounding of P~ switched off, the oracle's D matches sum_j P_ij dP_ij from the full
    matrices (P = softmax of the fake-quantised logits) to float32 accuracy; D from the FP4
    output O does not."""
    Q, K, V, dO = _inputs(192, 64, seed=6)
    fq = qat.fake_quant(Q, K, V)
    O, Op, L, _ = qat.qat_forward(fq, False, lambda a: a)
    _, _, P = fpa.fpa_forward(fq["Qf"], fq["Kf"], fq["Vf"], False)
    dP = np.asarray(dO, np.float64) @ np.swapaxes(fq["Vf"], -1, -2)
    want = (P * dP).sum(-1)
    D_op = (np.asarray(dO, np.float64) * Op).sum(-1)
    D_o = (np.asarray(dO, np.float64) * O).sum(-1)
    assert metrics.rel_l2(D_op, want) < 1e-6
    assert metrics.rel_l2(D_o, want) > 1e-2


@pytest.mark.parametrize("causal", [False, True])
def test_dv_is_the_gradient_of_the_forward_output(causal):
    """The forward's O is linear in V': O = W V' with W_ik = 2^(r_j(i) - M_i) phi(e_i, block j)_k /
    l_i (untiled, phi by grid search, j the key block of k).  The backward's dV must be W^T dO:
    the exact gradient of the fake-quantised forward (16-bit rounding of P^ switched off; the
    float32 roundings of L2 and of 2^(r - L2) leave ~1e-7)."""
    N, d = 192, 64
    Q, K, V, dO = _inputs(N, d, seed=7)
    Q, K, V, dO = Q[:, :1], K[:, :1], V[:, :1], dO[:, :1]
    ident = lambda a: a
    fq = qat.fake_quant(Q, K, V)
    O, Op, L, R = qat.qat_forward(fq, causal, ident)
    g = qat.qat_backward(fq, Op.astype(np.float32), L.astype(np.float32), R, dO, causal, ident)
    Qf, Kf, Vf = (fq[k][0, 0] for k in ("Qf", "Kf", "Vf"))
    c = float(np.float32(qat.LOG2E / math.sqrt(d)))
    W = np.zeros((N, N))
    for i in range(N):
        rs, ph, sums = {}, {}, {}
        for j in range(N // 64):
            keys = np.arange(64 * j, 64 * j + 64)
            valid = keys <= i if causal else np.ones(64, bool)
            if not valid.any():
                continue
            acc = Kf[keys] @ Qf[i]
            r = float(np.float32(np.where(valid, acc, -np.inf).max() * c))
            S = (acc * c).astype(np.float32)
            e = np.exp2(np.where(valid, (S - np.float32(r)).astype(np.float32), -np.inf).astype(np.float64)).astype(np.float32)
            rs[j], ph[j], sums[j] = r, _phi_brute(e), e.astype(np.float64).sum()
        M = max(rs.values())
        den = sum(2.0 ** (rs[j] - M) * sums[j] for j in rs)
        for j in rs:
            W[i, 64 * j:64 * j + 64] = 2.0 ** (rs[j] - M) * ph[j] / den
    assert metrics.rel_l2(O[0, 0], W @ Vf) < 1e-12
    assert metrics.rel_l2(g["dV"][0, 0], W.T @ np.asarray(dO[0, 0], np.float64)) < 1e-6


def test_straight_through_gradient_of_fake_quantised_operands():
    """With the backward's P fake quantisation and the 16-bit roundings switched off, the
    gradients are those of float64 attention evaluated at (Q', K', V'), to float32 accuracy."""
    Q, K, V, dO = _inputs(192, 64, seed=8)
    fq = qat.fake_quant(Q, K, V)
    ident = lambda a: a
    O, Op, L, R = qat.qat_forward(fq, True, ident)
    g = qat.qat_backward(fq, Op, L.astype(np.float32), R, dO, True, ident, bwd_p_quant=False)
    ref = fpa.fpa_backward(fq["Qf"], fq["Kf"], fq["Vf"], dO, True)
    for k in ("dQ", "dK", "dV"):
        assert metrics.rel_l2(g[k], ref[k]) < 1e-5, (k, metrics.rel_l2(g[k], ref[k]))
    # the method's dV carries the FP4 P and differs
    g_q = qat.qat_backward(fq, Op, L.astype(np.float32), R, dO, True, ident)
    assert metrics.rel_l2(g_q["dV"], ref["dV"]) > 1e-3


def test_ablation_d_from_fp4_output_is_worse():
    """Results (ablation): without the high-precision O' the gradients go wrong.  dQ and dK with D
    from the FP4 output O are further from the straight-through gradient than with D from O'."""
    Q, K, V, dO = _inputs(256, 64, seed=9)
    out = qat.run(Q, K, V, dO, False, workloads.round_fp16)
    fq = out["fq"]
    ref = fpa.fpa_backward(fq["Qf"], fq["Kf"], fq["Vf"], dO, False)
    bad = qat.qat_backward(fq, out["Op_stored"], out["L_stored"], out["R"], dO, False, workloads.round_fp16,
                           D_from=out["O_stored"])
    for k in ("dQ", "dK"):
        good_err = metrics.rel_l2(out[k], ref[k])
        bad_err = metrics.rel_l2(bad[k], ref[k])
        assert good_err < 1e-2 and bad_err > 3 * good_err, (k, good_err, bad_err)
