"""GPU parity of sage_quantize_smooth and sage_attn_fwd against the CPU oracle.

Bit-exact: int8 codes, block scales, mu_K / mu_Q, and the integer Q^ K^T block products (read from
the kernel's debug dump).  P codes: equal to the oracle's, or one apart where the oracle's
unrounded 127 * 2^x lies within the propagated rounding error of the half-integer between them
(tests/parity.py derives the bound), on at most 1e-3 of the entries.  P^ V^ products: the
oracle's where a tile's codes agree, else exactly the integer product of the kernel's own codes.
O: rel-l2 <= 1e-3 against the oracle's O rounded to the output type; L: max error <= 1e-4.
"""
import numpy as np
import pytest
import torch

from tests import parity
from tests.gpu_common import (causal_mask_full, fwd_dump_views, gpu_fwd, make_case, oracle_fwd,
                              rel_l2, to_dev, visited_blocks)

pytestmark = pytest.mark.gpu

CASES = [
    # N, d, dtype, causal, extra
    (128, 64, "fp16", False, {}),                                    # the tiny workload
    (320, 128, "fp16", True, {}),                                    # ragged tail, causal
    (384, 64, "bf16", True, dict(smooth_q=True)),                    # Q-smoothing bias
    (512, 128, "bf16", False, dict(qk="qknorm", k_offset_var=4.0)),  # QK-norm + K channel offsets
    (256, 128, "fp16", False, dict(sigma=5.0)),                      # large logits (sweep sigma 5)
    (192, 64, "fp16", False, dict(qk="outlier", smooth_q=True)),     # outlier channels
    (64, 128, "fp16", True, {}),                                     # one block: diagonal only
    (64, 64, "bf16", False, dict(smooth_q=True)),                    # one block, Q-smoothing
    (256, 128, "fp16", False, dict(sigma=10.0)),                     # the sweep's largest sigma
    (256, 64, "fp16", False, dict(special="const_k")),               # zero K blocks, s_K = 0
    (192, 128, "fp16", True, dict(special="const_k")),
]


def _ids(c):
    return f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}-{'-'.join(f'{k}={v}' for k, v in c[4].items())}"


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_quantize_bit_exact(case):
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    g = gpu_fwd(w, x)
    prep, _, _, _ = oracle_fwd(w, x, record=False)
    q = g["q"]
    for name in ("Qh", "Kh", "Vh"):
        assert np.array_equal(getattr(q, name).cpu().numpy(), prep[name]), name
    for name in ("sQ", "sK", "sV"):
        got = getattr(q, name).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), prep[name].view(np.uint32)), name
    assert np.array_equal(q.muK.cpu().numpy().view(np.uint32), prep["muK"].view(np.uint32))
    if w.smooth_q:
        assert np.array_equal(q.muQ.cpu().numpy().view(np.uint32), prep["muQ"].view(np.uint32))


# the quantiser alone on more blocks than its grid has CTAs: every CTA walks several blocks and
# reuses each of its shared-memory stages (8 at d = 64, 4 at d = 128); and bf16 blocks whose scale
# is subnormal in float32
QUANT_CASES = [
    # B, H, N, d, dtype, extra
    (1, 16, 4096, 64, "bf16", dict(smooth_q=True)),
    (2, 16, 2048, 128, "fp16", dict(k_offset_var=4.0)),
    (1, 16, 4096, 64, "fp16", dict(qk="outlier")),
    (1, 4, 1024, 128, "bf16", dict(special="tiny_qkv")),
    (1, 4, 1024, 64, "bf16", dict(special="tiny_qkv", smooth_q=True)),
]


@pytest.mark.parametrize("case", QUANT_CASES, ids=[f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}-{c[4]}-" + "-".join(f"{k}={v}" for k, v in c[5].items()) for c in QUANT_CASES])
def test_quantize_many_blocks_bit_exact(case):
    import bit_trainable_attention_sage_gb300 as sg
    from oracle import sage as osage
    B, H, N, d, dtype, extra = case
    w, x = make_case(N, d, dtype, False, B=B, H=H, **extra)
    Q, K, V = (to_dev(x[k], dtype) for k in ("Q", "K", "V"))
    q = sg.sage_quantize_smooth(Q, K, V, smooth_q=w.smooth_q)
    assert sg.sage_device_status() == 0
    prep = osage.prepare(x["Q"], x["K"], x["V"], smooth_q=w.smooth_q)
    for name in ("Qh", "Kh", "Vh"):
        assert np.array_equal(getattr(q, name).cpu().numpy(), prep[name]), name
    for name in ("sQ", "sK", "sV", "muK") + (("muQ",) if w.smooth_q else ()):
        got = getattr(q, name).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), np.asarray(prep[name], np.float32).view(np.uint32)), name
    if extra.get("special") == "tiny_qkv":
        s = np.concatenate([prep[k].ravel() for k in ("sQ", "sK", "sV")])
        assert np.any((s > 0) & (s < np.finfo(np.float32).tiny)), "no subnormal block scale"


def test_quantize_repeatable():
    """Ten quantise calls on the same inputs (every CTA waits for mu_K of the heads of its K blocks,
    which other CTAs finalise) give bit-identical codes, scales and means, equal to the oracle's."""
    import bit_trainable_attention_sage_gb300 as sg
    from oracle import sage as osage
    w, x = make_case(2048, 128, "fp16", False, B=2, H=16, k_offset_var=4.0)
    Q, K, V = (to_dev(x[k], "fp16") for k in ("Q", "K", "V"))
    prep = osage.prepare(x["Q"], x["K"], x["V"], smooth_q=False)
    for _ in range(10):
        q = sg.sage_quantize_smooth(Q, K, V)
        assert sg.sage_device_status() == 0
        for name in ("Qh", "Kh", "Vh"):
            assert np.array_equal(getattr(q, name).cpu().numpy(), prep[name]), name
        for name in ("sQ", "sK", "sV", "muK"):
            got = getattr(q, name).cpu().numpy()
            assert np.array_equal(got.view(np.uint32), np.asarray(prep[name], np.float32).view(np.uint32)), name


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_forward_parity(case):
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    g = gpu_fwd(w, x, dump=True)
    prep, O, L, rec = oracle_fwd(w, x)
    import workloads
    O_ref = workloads.round_to(O.astype(np.float32), dtype)
    O_gpu = g["O"].float().cpu().numpy()
    L_gpu = g["L"].cpu().numpy()
    assert np.all(np.isfinite(O_gpu)) and np.all(np.isfinite(L_gpu))
    assert rel_l2(O_gpu, O_ref) <= 1e-3
    assert np.max(np.abs(L_gpu - L)) <= 1e-4 * max(1.0, np.abs(L).max())
    S, P, PV = (t.cpu().numpy() for t in fwd_dump_views(g["dump"], w.B, w.H, N, d))
    mask = causal_mask_full(N) if causal else np.zeros((N, N), bool)
    n_codes = n_diff = 0
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            r = rec[(b, h)]
            for (i, j) in visited_blocks(N, causal):
                rows, cols = slice(64 * i, 64 * i + 64), slice(64 * j, 64 * j + 64)
                assert np.array_equal(S[b, h, rows, cols], r["S_int"][rows, cols]), (b, h, i, j)
                live = ~mask[rows, cols]
                St = r["S"][rows, cols].astype(np.float64)
                tile_r = np.where(live, St, -np.inf).max(axis=1, keepdims=True)
                tau = parity.fwd_code_tau(St, r["P_y"][rows, cols], np.where(np.isfinite(tile_r), tile_r, 0.0),
                                          r["acc_c"][rows, cols])
                nd, nl, dist = parity.check_flips(P[b, h, rows, cols], r["P_hat"][rows, cols],
                                                  r["P_y"][rows, cols], tau, live, (b, h, i, j))
                n_codes += nl
                n_diff += nd
                worst = max(worst, dist)
                assert np.all(P[b, h, rows, cols][~live] == 0)
                pc = P[b, h, rows, cols].astype(np.int64)
                want = r["PV_int"][(i, j)] if np.array_equal(pc, r["P_hat"][rows, cols]) \
                    else pc @ prep["Vh"][b, h, cols].astype(np.int64)
                assert np.array_equal(PV[b, h, i, j].astype(np.int64), want), (b, h, i, j)
    print(f"\n{_ids(case)}: P code flips {n_diff}/{n_codes} (largest distance of a flip from its "
          f"half-integer {worst:.2e}), O rel-l2 {rel_l2(O_gpu, O_ref):.2e}, "
          f"L max err {np.max(np.abs(L_gpu - L)):.2e}")
    assert n_diff <= 1e-3 * n_codes, (n_diff, n_codes)
