"""GPU parity of sage_attn_bwd against the CPU oracle, through the C ABI.

Bit-exact: the dO^ codes and block scales; the recomputed integer Q^ K^T products; the integer
block products P^T dO^ (dV), dS^ K^ (dQ) and dS^T Q^ (dK) of every tile whose codes agree with the
oracle's (for a tile with a flipped code: the exact integer product of the kernel's own codes).
P and dS codes: equal to the oracle's, or one apart where the oracle's unrounded value lies within
the propagated rounding error of the half-integer between them (tests/parity.py derives the
bound); such flips on at most 1e-3 of the codes.  Tile scales within the same propagated error.
dP: within the float32 accumulation bound of the exact product.  dQ, dK, dV: rel-l2 <= 1e-3 over
the whole tensor and <= 5e-3 over every 64-row block.  Degenerate inputs: equal keys (zero K
blocks), dO = 0 (every dS tile zero), dS tiles on both sides of the 2^-120 zero-tile bound,
sigma = 10 logits, and the tiny workload with dO ~ N(0, 1).
"""
import numpy as np
import pytest

from tests import parity
from tests.gpu_common import causal_mask_full, gpu_run, make_case, oracle_run, rel_l2, visited_blocks

pytestmark = pytest.mark.gpu

CASES = [
    (128, 64, "fp16", False, dict(do_var=1.0)),                      # the tiny workload
    (320, 128, "fp16", True, {}),
    (384, 64, "bf16", True, dict(smooth_q=True)),
    (512, 128, "bf16", False, dict(qk="qknorm", k_offset_var=4.0, do_var=1e-4)),
    (256, 128, "fp16", False, dict(sigma=5.0)),
    (256, 128, "fp16", False, dict(sigma=10.0)),                     # the sweep's largest sigma
    (192, 64, "fp16", True, dict(qk="outlier", smooth_q=True)),
    (64, 128, "fp16", True, {}),                                     # one block: diagonal only
    (64, 64, "bf16", False, dict(smooth_q=True)),                    # one block, Q-smoothing
    (256, 64, "fp16", False, dict(special="const_k")),               # zero K blocks, s_K = 0
    (192, 128, "fp16", True, dict(special="const_k")),
    (256, 128, "fp16", False, dict(special="zero_do")),              # every dS tile zero
    (256, 64, "bf16", False, dict(special="tiny_ds", do_var=1.0)),   # dS around 2^-120
]

FLIP_RATE = 1e-3


def _ids(c):
    return f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}-{'-'.join(f'{k}={v}' for k, v in c[4].items())}"


def compare_backward(w, x, g, ref):
    """Every check of the module docstring on one problem; returns the measured statistics."""
    N, d = w.N, w.d
    stats = {}
    for k in ("dQ", "dK", "dV"):
        assert np.all(np.isfinite(g[k])), k
        stats[k] = rel_l2(g[k], ref[k])
        stats[k + "_block"] = parity.block_rel_l2(g[k], ref[k])
        assert stats[k] <= 1e-3, (k, stats[k])
        assert stats[k + "_block"] <= 5e-3, (k, stats[k + "_block"])
    dmp = g["dump"]
    prep = ref["prep"]
    assert np.array_equal(dmp["dOh"], ref["dOh"])
    assert np.array_equal(dmp["sdO"].view(np.uint32), ref["sdO"].view(np.uint32))
    # D is formed from the kernel's own stored O (its 16-bit rounding differs from the oracle's)
    D_own = (x["dO"].astype(np.float64) * g["O"].astype(np.float64)).sum(-1)
    assert rel_l2(dmp["D"], D_own) <= 1e-5
    assert rel_l2(dmp["D"], ref["D"]) <= 1e-3
    L2_ref = parity.l2_of(ref["L_stored"])
    L2_gpu = parity.l2_of(g["L"])
    mask = causal_mask_full(N) if w.causal else np.zeros((N, N), bool)
    rec = ref["record"]
    n_live = flips_p = flips_ds = 0
    worst = dict(p=0.0, ds=0.0, dp=0.0)
    exact_tiles = own_tiles = 0
    for b in range(w.B):
        for h in range(w.H):
            r = rec[(b, h)]
            dO64 = np.abs(x["dO"][b, h].astype(np.float64))
            V64 = np.abs(x["V"][b, h].astype(np.float64))
            for (i, j) in visited_blocks(N, w.causal):
                rows, cols = slice(64 * i, 64 * i + 64), slice(64 * j, 64 * j + 64)
                live = ~mask[rows, cols]
                # recomputed S: bit-exact
                assert np.array_equal(dmp["S"][b, h, rows, cols][live], r["S_int"][rows, cols][live]), (b, h, i, j)
                # dP: float32 accumulation of exact 16-bit products
                absdp = dO64[rows] @ V64[cols].T
                ddp = np.abs(dmp["dP"][b, h, rows, cols].astype(np.float64) - r["dP"][rows, cols])
                bound = 2 * (d + 2) * parity.U * absdp
                assert np.all(ddp[live] <= bound[live]), (b, h, i, j, "dP")
                worst["dp"] = max(worst["dp"], float((ddp / np.maximum(bound, 1e-300))[live].max(initial=0)))
                # codes and scales
                sp_o, sds_o = float(r["sP"][i, j]), float(r["sdS"][i, j])
                sp_g, sds_g = float(dmp["sP"][b, h, i, j]), float(dmp["sdS"][b, h, i, j])
                P_est = r["P_y"][rows, cols].astype(np.float64) * sp_o
                tau_p, tau_ds, eps_sp, eps_sds = parity.bwd_tile_taus(
                    r["S_bwd"][rows, cols], r["acc_c_bwd"][rows, cols], L2_ref[b, h, rows], L2_gpu[b, h, rows], P_est,
                    r["dP"][rows, cols], ref["D"][b, h, rows], dmp["D"][b, h, rows], absdp,
                    r["P_y"][rows, cols], r["dS_y"][rows, cols], d, live)
                for what, s_o, s_g, eps in (("sP", sp_o, sp_g, eps_sp), ("sdS", sds_o, sds_g, eps_sds)):
                    if s_o == 0 or s_g == 0:
                        assert s_o == s_g, (what, b, h, i, j, s_o, s_g)
                    else:
                        assert abs(s_g / s_o - 1) <= parity.SAFETY * eps, (what, b, h, i, j, s_o, s_g)
                fp, nl, dist_p = parity.check_flips(dmp["P"][b, h, rows, cols], r["P_hat"][rows, cols],
                                                    r["P_y"][rows, cols], tau_p, live, ("P", b, h, i, j))
                fd, _, dist_ds = parity.check_flips(dmp["dS"][b, h, rows, cols], r["dS_hat"][rows, cols],
                                                    r["dS_y"][rows, cols], tau_ds, live, ("dS", b, h, i, j))
                assert np.all(dmp["P"][b, h, rows, cols][~live] == 0) and np.all(dmp["dS"][b, h, rows, cols][~live] == 0)
                flips_p += fp
                flips_ds += fd
                n_live += nl
                worst["p"] = max(worst["p"], dist_p)
                worst["ds"] = max(worst["ds"], dist_ds)
                # block products: the oracle's where the codes agree, else those of the kernel's codes
                pc = dmp["P"][b, h, rows, cols].astype(np.int64)
                dc = dmp["dS"][b, h, rows, cols].astype(np.int64)
                same_p = np.array_equal(pc, r["P_hat"][rows, cols])
                same_d = np.array_equal(dc, r["dS_hat"][rows, cols])
                want_dv = r["dV_int"][(i, j)] if same_p else pc.T @ dmp["dOh"][b, h, rows].astype(np.int64)
                want_dq = r["dQ_int"][(i, j)] if same_d else dc @ prep["Kh"][b, h, cols].astype(np.int64)
                want_dk = r["dK_int"][(i, j)] if same_d else dc.T @ prep["Qh"][b, h, rows].astype(np.int64)
                assert np.array_equal(dmp["dV_int"][b, h, i, j].astype(np.int64), want_dv), (b, h, i, j, "dV")
                assert np.array_equal(dmp["dQ_int"][b, h, i, j].astype(np.int64), want_dq), (b, h, i, j, "dQ")
                assert np.array_equal(dmp["dK_int"][b, h, i, j].astype(np.int64), want_dk), (b, h, i, j, "dK")
                exact_tiles += int(same_p) + int(same_d)
                own_tiles += int(not same_p) + int(not same_d)
    stats.update(flips_p=flips_p, flips_ds=flips_ds, codes=n_live, worst_flip_dist_p=worst["p"],
                 worst_flip_dist_ds=worst["ds"], dp_bound_use=worst["dp"], exact_tiles=exact_tiles,
                 own_code_tiles=own_tiles)
    assert flips_p <= FLIP_RATE * n_live, (flips_p, n_live)
    assert flips_ds <= FLIP_RATE * n_live, (flips_ds, n_live)
    return stats


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_backward_parity(case):
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    g = gpu_run(w, x, dump=True)
    ref = oracle_run(w, x, products=True)
    st = compare_backward(w, x, g, ref)
    if extra.get("special") == "tiny_ds":
        # the case must put tiles on both sides of the zero-tile bound, near it
        maxima = np.concatenate([ref["record"][k]["sdS"].ravel() for k in ref["record"]]) * 127.0
        assert np.any((maxima >= 2.0 ** -120) & (maxima < 2.0 ** -117)), "no tile just above 2^-120"
        assert np.any((maxima == 0) | ((maxima < 2.0 ** -120))), "no zero tile"
    if extra.get("special") == "zero_do":
        for k in ("dQ", "dK", "dV"):
            assert not g[k].any(), k
    print(f"\n{_ids(case)}: " + ", ".join(f"{k} {v:.3g}" if isinstance(v, float) else f"{k} {v}" for k, v in st.items()))
