"""Pins for the SageBwd oracle's forward and backward (CPU only).

* Dequantised limit: the oracle's tiled code, run with every quantiser replaced by the identity
  and no float32 rounding, must equal float64 FPA (itself pinned by finite differences).  This
  pins the tiling, the online softmax of "SageAttention3 ..." (review) eq. (1), the s_P rescaling of
  eq. (8), L, D and the backward steps of the structured summary's method steps.
* Closed form: the quantised forward is independent of the order of the key blocks,
  O_i = sum_j 2^(r_ij - M_i) (s_V,j / 127) P^_ij V^_j / sum_j sum_k 2^(t_ijk - M_i).
* Special cases with known answers, exact integer products, the tile quantiser against an exact
  rational re-derivation, and the trend of the pages' Table 1 ("SageBwd: A Trainable Low-bit
  Attention", Table 1 -- exact values unpinned: N, d and block sizes are not printed).
"""
import math
from fractions import Fraction as Fr

import numpy as np
import pytest

import workloads
from oracle import sage, fpa, metrics, quant
from tests.exact import fl32, rne


def _inputs(N, d, seed, B=1, H=2, scale=1.0, k_offset=0.0, dtype="fp16"):
    rng = np.random.default_rng(seed)
    shp = (B, H, N, d)
    Q, K, V, dO = (rng.standard_normal(shp).astype(np.float32) for _ in range(4))
    Q *= np.float32(scale)
    K = K * np.float32(scale) + np.float32(k_offset)
    dO *= np.float32(0.1)
    r = workloads.round_fp16 if dtype == "fp16" else workloads.round_bf16
    return r(Q), r(K), r(V), r(dO)


@pytest.mark.parametrize("N,d,causal,smooth_k,smooth_q", [
    (256, 64, False, True, False),
    (256, 64, True, True, False),
    (192, 128, True, True, True),
    (128, 64, False, False, False),
    (256, 32, True, False, True),
])
def test_dequantised_limit_equals_fpa(N, d, causal, smooth_k, smooth_q):
    Q, K, V, dO = _inputs(N, d, seed=N + d, k_offset=2.0)
    out = sage.run(Q, K, V, dO, causal, lambda a: a, smooth_k=smooth_k, smooth_q=smooth_q,
                   arith=sage.DEQUANTISED)
    O, _, _ = fpa.fpa_forward(Q, K, V, causal)
    g = fpa.fpa_backward(Q, K, V, dO, causal)
    assert metrics.rel_l2(out["O"], O) < 1e-12
    for k in ("dQ", "dK", "dV"):
        assert metrics.rel_l2(out[k], g[k]) < 1e-12, k
    assert metrics.rel_l2(out["D"], g["D"]) < 1e-12
    # L is the log-sum-exp of the logits actually formed: with K-smoothing, those of K - mu_K
    Kref = K - K.astype(np.float64).mean(axis=-2, keepdims=True) if smooth_k else K
    L_ref = fpa.fpa_forward(Q, Kref, V, causal)[1]
    assert np.max(np.abs(out["L"] - L_ref)) < 1e-11


def _closed_form_O(prep, causal):
    """Order-independent closed form of the quantised forward, evaluated row by row:
    O_i = sum_j 2^(r_ij - M_i) (s_V,j / 127) P^_ij V^_j / sum_j 2^(r_ij - M_i) sum_k 2^(x_ijk),
    with the per-tile codes P^ = rint(127 * 2^x), x = fl32(S - r), S = fl32(acc c), r = max S."""
    Qh, Kh, Vh, sQ, sK, sV = (prep[k] for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV"))
    B, H, N, d = Qh.shape
    T = N // 64
    sl2 = np.float32(sage.LOG2E / math.sqrt(d))
    O = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            acc = np.einsum("nc,mc->nm", Qh[b, h].astype(np.int64), Kh[b, h].astype(np.int64)).astype(np.float64)
            c = ((np.repeat(sQ[b, h], 64)[:, None] * np.repeat(sK[b, h], 64)[None, :]).astype(np.float32) * sl2).astype(np.float64)
            valid = ~np.triu(np.ones((N, N), bool), 1) if causal else np.ones((N, N), bool)
            accj = acc.reshape(N, T, 64)
            cj = c.reshape(N, T, 64)[:, :, 0]
            vj = valid.reshape(N, T, 64)
            live = vj.any(axis=2)
            amax = np.where(vj, accj, -np.inf).max(axis=2)
            r = np.where(live, (np.where(live, amax, 0) * cj).astype(np.float32), -np.inf)
            Sj = (accj * cj[:, :, None]).astype(np.float32)
            x = (Sj - np.where(live, r, 0)[:, :, None].astype(np.float32)).astype(np.float32)
            x = np.where(vj, x, -np.inf)
            e64 = np.exp2(x.astype(np.float64))
            p_hat = np.rint(np.float32(127) * e64.astype(np.float32))
            r64 = r.astype(np.float64)
            Mrow = r64.max(axis=1)
            w = np.where(live, np.exp2(np.where(live, r64, 0.0) - Mrow[:, None]), 0.0)
            num = np.zeros((N, d))
            for j in range(T):
                num += (w[:, j] / 127.0 * sV[b, h, j])[:, None] * (p_hat[:, j, :] @ Vh[b, h, 64 * j:64 * j + 64].astype(np.float64))
            den = (w * e64.sum(axis=2)).sum(axis=1)
            O[b, h] = num / den[:, None]
    return O


@pytest.mark.parametrize("causal", [False, True])
def test_quantised_forward_closed_form(causal):
    Q, K, V, _ = _inputs(256, 64, seed=11, scale=2.0)
    prep = sage.prepare(Q, K, V)
    O, L = sage.sage_forward(prep, causal)
    Oc = _closed_form_O(prep, causal)
    assert metrics.rel_l2(O, Oc) < 1e-12


def test_integer_products_exact():
    Q, K, V, _ = _inputs(128, 64, seed=5)
    prep = sage.prepare(Q, K, V)
    rec = {}
    sage.sage_forward(prep, False, record=rec)
    for (b, h), r in rec.items():
        want = np.einsum("nc,mc->nm", prep["Qh"][b, h].astype(np.int64), prep["Kh"][b, h].astype(np.int64))
        assert np.array_equal(r["S_int"], want)
        for (i, j), pv in r["PV_int"].items():
            want = r["P_hat"][64 * i:64 * i + 64, 64 * j:64 * j + 64] @ prep["Vh"][b, h, 64 * j:64 * j + 64].astype(np.int64)
            assert np.array_equal(pv, want)
    # the extreme case: every code +-127 over a 128-long contraction stays exact
    a = np.full((64, 128), 127, np.int64)
    a[1] = -127
    p = sage.QUANTISED.int_mm(a, a.T)
    assert p[0, 0] == 128 * 127 * 127 == 2064512 and p[0, 1] == -2064512


def test_token_quantiser():
    x = np.array([[0.0, -1.0, -0.5, -np.inf, -30.0]], np.float32)
    e64, q = sage.QUANTISED.token_quant(x)
    assert q.tolist() == [[127, 64, 90, 0, 0]]    # 127, 63.5 -> 64 (even), 127/sqrt(2) = 89.8
    assert e64[0, 0] == 1.0 and e64[0, 3] == 0.0


def test_tile_quantiser_against_exact_rationals():
    rng = np.random.default_rng(3)
    for scale in (1.0, 1e-7, 1e-30, 3e-37):
        x = (rng.standard_normal((64, 64)) * scale).astype(np.float32)
        s, q = sage.QUANTISED.tile_quant(x)
        mx = max(abs(Fr(float(v))) for v in x.ravel())
        if mx < Fr(2) ** -120:
            assert s == 0 and not q.any()
            continue
        se = fl32(mx / 127)
        inv = fl32(1 / se)
        assert Fr(float(s)) == se
        # the float32 product x * inv, then the nearest integer (ties to even), clamped
        qe = [max(-127, min(127, rne(fl32(Fr(float(v)) * inv)))) for v in x.ravel()]
        assert q.ravel().tolist() == qe
        assert max(abs(v) for v in qe) == 127
    s, q = sage.QUANTISED.tile_quant(np.zeros((64, 64), np.float32))
    assert s == 0 and not q.any()


def test_tile_quantiser_rounding_boundaries():
    """Hand-worked: max = 127 gives s = 1 and inv = 1 exactly, so the codes are x rounded to the
    nearest integer, ties to even: 62.5 -> 62, 63.5 -> 64, -2.5 -> -2, 0.49999997 -> 0, and
    63.5 - 2^-15 (a float32 value) -> 63: one rounding, not a rounding to a coarser grid first."""
    x = np.zeros((64, 64), np.float32)
    x.ravel()[:6] = [127.0, 62.5, 63.5, -2.5, 63.5 - 2.0 ** -15, 0.49999997]
    s, q = sage.QUANTISED.tile_quant(x)
    assert s == np.float32(1.0)
    assert q.ravel()[:6].tolist() == [127, 62, 64, -2, 63, 0]


def test_special_case_constant_keys():
    """All K rows equal: K-smoothing makes K_sm = 0, every K block a zero block, S = 0, so every
    P^ code is 127 and O is the mean over keys of the dequantised V (non-causal)."""
    Q, K, V, _ = _inputs(256, 64, seed=9)
    K = np.broadcast_to(K[:, :, :1, :], K.shape).copy()
    prep = sage.prepare(Q, K, V)
    assert not prep["Kh"].any() and not prep["sK"].any()
    rec = {}
    O, L = sage.sage_forward(prep, False, record=rec)
    assert np.all(rec[(0, 0)]["P_hat"] == 127)
    Vdeq = prep["Vh"].astype(np.float64) * np.repeat(prep["sV"], 64, axis=2)[..., None]
    assert np.allclose(O, Vdeq.mean(axis=2, keepdims=True), rtol=1e-13, atol=1e-15)
    assert np.allclose(L, math.log(256), rtol=1e-14)


def test_special_case_causal_first_row():
    """Causal row 0 sees key 0 only: its logit is the tile's row max r, so x = fl32(S - r) = 0, its
    code is 127 and s_P = 1/127, hence O_0 = s_V,0 V^_0 exactly."""
    Q, K, V, _ = _inputs(128, 64, seed=10)
    prep = sage.prepare(Q, K, V)
    O, L = sage.sage_forward(prep, True)
    want = prep["sV"][:, :, 0, None].astype(np.float64) * prep["Vh"][:, :, 0, :]
    assert np.array_equal(O[:, :, 0, :], want)


def test_backward_dp_is_unquantised_and_tiles_bounded():
    """dP is formed from the 16-bit dO and V (Table 2 of the pages shows dP at cos 1.0000 / rel
    0.0000), and the per-tile codes reconstruct P and dS within half a step."""
    Q, K, V, dO = _inputs(128, 64, seed=12)
    rec = {}
    out = sage.run(Q, K, V, dO, False, workloads.round_fp16, record=rec)
    g = fpa.fpa_backward(Q, K, V, dO, False, O=out["O_stored"].astype(np.float64))
    r = rec[(0, 0)]
    assert metrics.rel_l2(r["dP"], g["dP"][0, 0]) < 1e-6
    assert metrics.cos_sim(r["P"], g["P"][0, 0]) > 0.99
    assert metrics.cos_sim(r["dS"], g["dS"][0, 0]) > 0.9


def test_sweep_trend_matches_table1():
    """Errors vs FPA grow with sigma_Q = sigma_K and hit dQ, dK hardest ("SageBwd: A Trainable
    Low-bit Attention", Table 1: at sigma 10, dQ/dK cos ~0.78 and rel-l2 ~0.66, O/dV cos >= 0.99)."""
    rows = []
    for sigma in (1.0, 5.0, 10.0):
        w = workloads.get("sweep", sigma=sigma, N=512)
        x = workloads.make_inputs(w, heads=1)
        out = sage.run(x["Q"], x["K"], x["V"], x["dO"], False, workloads.round_fp16)
        O, _, _ = fpa.fpa_forward(x["Q"], x["K"], x["V"])
        g = fpa.fpa_backward(x["Q"], x["K"], x["V"], x["dO"])
        rows.append({k: metrics.rel_l2(out[k], ref) for k, ref in
                     (("O", O), ("dQ", g["dQ"]), ("dK", g["dK"]), ("dV", g["dV"]))})
        rows[-1]["cos_dQ"] = metrics.cos_sim(out["dQ"], g["dQ"])
    for k in ("O", "dQ", "dK", "dV"):
        assert rows[0][k] < rows[1][k] < rows[2][k], k
    assert rows[0]["O"] < 0.05 and rows[0]["dQ"] < 0.1
    last = rows[2]
    assert last["dQ"] > 3 * last["O"] and last["dK"] > 3 * last["dV"]
    assert 0.4 < last["dQ"] < 0.9 and 0.6 < last["cos_dQ"] < 0.95


def _exact_code_tensor(rng, shape, log2_step):
    """Integer codes in [-127, 127] with a 127 in every 64-token block, times 2^log2_step: the
    per-block quantiser returns exactly these codes with the scale 2^log2_step."""
    codes = rng.integers(-127, 128, size=shape).astype(np.float64)
    codes[..., ::64, 0] = 127.0
    return (codes * 2.0 ** log2_step).astype(np.float32)


def test_dp_int8_equals_16bit_dp_when_codes_are_exact():
    """INT8-dP ablation ("SageAttention3 ..." (review), Table 1c): when V and dO are exactly their
    codes times power-of-two block scales, dP = fl32(MM(dO^, V^T) fl32(s_dO s_V)) equals the 16-bit
    product, so every gradient must come out bit for bit the same as the method's path.  A dropped
    scale, a transposed operand or a wrong block index breaks the equality."""
    rng = np.random.default_rng(21)
    B, H, N, d = 1, 2, 192, 64
    Q, K = (workloads.round_fp16(rng.standard_normal((B, H, N, d)).astype(np.float32)) for _ in range(2))
    V = _exact_code_tensor(rng, (B, H, N, d), -3)
    dO = _exact_code_tensor(rng, (B, H, N, d), -9)
    for causal in (False, True):
        a = sage.run(Q, K, V, dO, causal, workloads.round_fp16)
        b = sage.run(Q, K, V, dO, causal, workloads.round_fp16, dp_int8=True)
        for k in ("dQ", "dK", "dV"):
            assert np.array_equal(a[k], b[k]), (causal, k)


def test_dp_int8_ablation_is_less_accurate():
    """Table 1c of "SageAttention3 ..." (review): forming dO V^T from INT8 codes (cos 97.47 %) is
    worse than keeping it in 16 bits (cos 99.77 %).  On Gaussian inputs the oracle's INT8-dP dP
    and dQ, dK must be further from FPA than the method's."""
    Q, K, V, dO = _inputs(256, 64, seed=33)
    g = fpa.fpa_backward(Q, K, V, dO, False)
    errs = {}
    for flag in (False, True):
        rec = {}
        out = sage.run(Q, K, V, dO, False, workloads.round_fp16, record=rec, dp_int8=flag)
        errs[flag] = dict(dP=metrics.rel_l2(rec[(0, 0)]["dP"], g["dP"][0, 0]),
                          dQ=metrics.rel_l2(out["dQ"], g["dQ"]), dK=metrics.rel_l2(out["dK"], g["dK"]))
    assert errs[False]["dP"] < 1e-5 < errs[True]["dP"]
    assert errs[True]["dQ"] > errs[False]["dQ"] and errs[True]["dK"] > errs[False]["dK"]
