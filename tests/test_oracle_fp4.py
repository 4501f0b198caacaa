"""Pins of the oracle's SageAttention3 FP4 forward ("SageAttention3 ..." (review), eq. (2)-(6):
NVFP4 microscaling -- E2M1 values, 1 x 16 blocks, E4M3 scales -- and the two-level P scaling),
independent of the oracle's own rounding code: brute-force nearest points of the decoded grids,
exact rationals, a closed form of the forward, and the pages' accuracy ordering."""
from __future__ import annotations

import math
from fractions import Fraction as Fr

import numpy as np
import pytest

import workloads
from oracle import fp4, fpa, metrics, quant
from tests.exact import fl32


def _nearest(y, vals, pats):
    """Nearest grid value (grid = non-negative values with their bit patterns), ties to the even
    pattern; values beyond the grid take its largest point."""
    y = np.asarray(y, np.float64).ravel()
    dist = np.abs(np.abs(y)[:, None] - vals[None, :])
    tie = dist == dist.min(axis=1, keepdims=True)
    score = np.where(tie, 2 - (pats[None, :] % 2 == 0), 9)
    return np.copysign(vals[np.argmin(score, axis=1)], y)


E2M1_VALS = fp4.e2m1_decode(np.arange(8))
E2M1_PATS = np.arange(8)
E4M3_VALS = quant.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
E4M3_PATS = np.arange(0x7F)


def test_e2m1_decode_and_grid():
    assert fp4.e2m1_decode(np.arange(16)).tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                                                      -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_rounding_against_brute_force():
    mids = (E2M1_VALS[1:] + E2M1_VALS[:-1]) / 2
    rng = np.random.default_rng(1)
    y = np.concatenate([E2M1_VALS, mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                        rng.uniform(0, 9, 5000), [6.0, 6.5, 7.0, 100.0]])
    y = np.concatenate([y, -y]).astype(np.float32).astype(np.float64)
    assert np.array_equal(fp4.e2m1_round(y), _nearest(y, E2M1_VALS, E2M1_PATS))


def test_block_quantiser_hand_worked():
    """[1, -3, 0.4, 12, 0...]: s = e4m3(12/6) = 2, codes [0.5, -1.5, 0 (0.2 < 0.25), 6].
    [7, 1, 0...]: 7/6 = 1.1667 -> E4M3 1.125 (spacing 1/8), 7/1.125 = 6.2 saturates to 6,
    1/1.125 = 0.89 -> 1."""
    q, s = fp4.nvfp4_quant(np.array([[1.0, -3.0, 0.4, 12.0] + [0.0] * 12], np.float32))
    assert s.tolist() == [[2.0]] and q[0, :4].tolist() == [0.5, -1.5, 0.0, 6.0]
    q, s = fp4.nvfp4_quant(np.array([[7.0, 1.0] + [0.0] * 14], np.float32))
    assert s.tolist() == [[1.125]] and q[0, :2].tolist() == [6.0, 1.0]
    q, s = fp4.nvfp4_quant(np.zeros((1, 16), np.float32))
    assert s.tolist() == [[0.0]] and not q.any()


def test_block_quantiser_against_exact_rationals():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((8, 64)) * np.exp(rng.normal(0, 2, (8, 1)))).astype(np.float32)
    q, s = fp4.nvfp4_quant(x, axis=-1)
    for r in range(8):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16]
            mx = max(abs(Fr(float(v))) for v in blk)
            se = _nearest([float(fl32(mx / 6))], E4M3_VALS, E4M3_PATS)[0]
            assert s[r, b] == se
            if se == 0:
                assert not q[r, 16 * b:16 * b + 16].any()
                continue
            want = _nearest([float(fl32(Fr(float(v)) / Fr(float(se)))) for v in blk], E2M1_VALS, E2M1_PATS)
            assert np.array_equal(q[r, 16 * b:16 * b + 16].astype(np.float64), want)


def test_v_is_blocked_along_tokens():
    rng = np.random.default_rng(3)
    V = rng.standard_normal((1, 1, 64, 32)).astype(np.float32)
    q, s = fp4.nvfp4_quant(V, axis=-2)
    assert s.shape == (1, 1, 4, 32)
    for blk in range(4):
        qb, sb = fp4.nvfp4_quant(V[0, 0, 16 * blk:16 * blk + 16, 5][None, :])
        assert sb[0, 0] == s[0, 0, blk, 5]
        assert np.array_equal(qb[0], q[0, 0, 16 * blk:16 * blk + 16, 5])


def _inputs(N, d, seed, q_off=0.0, k_off=0.0):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((1, 1, N, d)) + q_off * rng.standard_normal((1, 1, 1, d))
    K = rng.standard_normal((1, 1, N, d)) + k_off * rng.standard_normal((1, 1, 1, d))
    V = rng.standard_normal((1, 1, N, d))
    r = workloads.round_fp16
    return r(Q.astype(np.float32)), r(K.astype(np.float32)), r(V.astype(np.float32))


@pytest.mark.parametrize("causal", [False, True])
def test_fp4_forward_closed_form(causal):
    """O_i = sum_j 2^(r_ij - M_i) / 2688 (P'_ij V'_j) / sum_j 2^(r_ij - M_i) sum_k 2^(x_ijk), with
    x = fl32(fl32(acc c) - r) and P' the brute-force NVFP4 of fl32(2688 fl32(2^x)) per 16 keys,
    evaluated without tiling."""
    N, d = 192, 64
    Q, K, V = _inputs(N, d, seed=4)
    prep = fp4.quantize_fp4(Q, K, V)
    O, _ = fp4.sage_fp4_forward(prep, causal)
    Qd = fp4.dequant(prep["Qc"], prep["sQ"])[0, 0]
    Kd = fp4.dequant(prep["Kc"], prep["sK"])[0, 0]
    Vd = fp4.dequant(prep["Vc"], prep["sV"], axis=-2)[0, 0]
    c = float(np.float32(1.4426950408889634 / math.sqrt(d)))
    T = N // 64
    acc = Qd @ Kd.T
    valid = ~np.triu(np.ones((N, N), bool), 1) if causal else np.ones((N, N), bool)
    num = np.zeros((N, d))
    den = np.zeros(N)
    rmax = np.full(N, -np.inf)
    per = []
    for j in range(T):
        a = acc[:, 64 * j:64 * j + 64]
        vj = valid[:, 64 * j:64 * j + 64]
        live = vj.any(axis=1)
        r = np.where(live, (np.where(vj, a, -np.inf).max(axis=1) * c).astype(np.float32), -np.inf)
        S = (a * c).astype(np.float32)
        x = np.where(vj, (S - np.where(live, r, 0)[:, None].astype(np.float32)).astype(np.float32), -np.inf)
        e = np.exp2(x.astype(np.float64))
        v = (np.float32(2688) * e.astype(np.float32)).astype(np.float32)
        pd = np.zeros_like(e)
        for g in range(4):
            vb = v[:, 16 * g:16 * g + 16]
            s2 = _nearest((vb.max(axis=1) / np.float32(6)).astype(np.float32), E4M3_VALS, E4M3_PATS)
            inv = np.where(s2 == 0, 0, (np.float32(1) / np.where(s2 == 0, 1, s2).astype(np.float32)))
            codes = _nearest((vb * inv.astype(np.float32)[:, None]).astype(np.float32), E2M1_VALS, E2M1_PATS).reshape(vb.shape)
            pd[:, 16 * g:16 * g + 16] = codes * s2[:, None]
        per.append((r.astype(np.float64), e, pd))
        rmax = np.maximum(rmax, r.astype(np.float64))
    for j, (r, e, pd) in enumerate(per):
        w = np.where(np.isfinite(r), np.exp2(np.where(np.isfinite(r), r, 0) - rmax), 0.0)
        num += (w / 2688.0)[:, None] * (pd @ Vd[64 * j:64 * j + 64])
        den += w * e.sum(axis=1)
    assert metrics.rel_l2(O[0, 0], num / den[:, None]) < 1e-12


def test_fp4_less_accurate_than_int8_and_smoothing_helps():
    """FP4 trails INT8 against full precision; with channel offsets on Q and K, smoothing both
    ("SageAttention3 ..." (review): Q+K smoothing lifts FP4 CosSim from 0.9156 to 0.9912)
    brings FP4 closer to full precision than no smoothing."""
    from oracle import sage as osage
    Q, K, V = _inputs(256, 64, seed=5)
    O_ref, _, _ = fpa.fpa_forward(Q, K, V, False)
    O4, _ = fp4.sage_fp4_forward(fp4.quantize_fp4(Q, K, V), False)
    prep8 = osage.prepare(Q, K, V)
    O8, _ = osage.sage_forward(prep8, False)
    assert metrics.rel_l2(O4, O_ref) > metrics.rel_l2(O8, O_ref)
    Q, K, V = _inputs(256, 64, seed=6, q_off=4.0, k_off=8.0)
    O_ref, _, _ = fpa.fpa_forward(Q, K, V, False)
    plain, _ = fp4.sage_fp4_forward(fp4.quantize_fp4(Q, K, V, smooth_k=False, smooth_q=False), False)
    smooth, _ = fp4.sage_fp4_forward(fp4.quantize_fp4(Q, K, V, smooth_k=True, smooth_q=True), False)
    assert metrics.rel_l2(smooth, O_ref) < metrics.rel_l2(plain, O_ref)
