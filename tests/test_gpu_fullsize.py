"""GPU parity at the full sizes of the benchmarked workloads, in the launch configuration the
benchmark times (one quantise, forward and backward call over the whole batch).

The CUDA path runs on the full tensors; the oracle recomputes a sample it can afford: every code,
block scale and mean bit for bit (the whole tensors), and O, L, dQ, dK, dV on the rows of sampled
query and key blocks of one head, within rel-l2 1e-3.  The oracle's rows need the log-sum-exp and D
of every query row their tiles touch: for the non-causal headline that is a full forward of the
sampled head; for causal workloads the sampled blocks sit at the two ends of the sequence, where
only a few query blocks are involved.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import sage as osage
from tests.gpu_common import rel_l2, to_dev

pytestmark = pytest.mark.gpu

# (workload, overrides, sampled head (b, h), forward query blocks, dQ blocks, dK/dV blocks);
# None for the forward blocks means the whole head (non-causal: every row's L and D is needed)
CASES = [
    ("headline", {}, (1, 5), None, [0, 77], [5, 100]),
    ("qknorm", {}, (3, 11), "ends", [0, 1, -1], [-1, -2]),
    ("outlier", dict(smooth_q=True), (1, 30), "ends", [0, 2, -1], [-1, -2]),
    ("longseq", {}, (0, 3), "ends", [0, 1, -1], [-1, -2]),
]


def _run_gpu(w, x):
    import bit_trainable_attention_sage_gb300 as sg
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    q = sg.sage_quantize_smooth(Q, K, V, smooth_q=w.smooth_q)
    Kb = K if w.smooth_q else None
    O, L = sg.sage_attn_fwd(q, causal=w.causal, K=Kb)
    dQ, dK, dV = sg.sage_attn_bwd(q, V, O, L, dO, causal=w.causal, K=Kb)
    st = sg.sage_device_status()
    assert st == 0, sg.sage_status_string(st)
    return q, O, L, dQ, dK, dV


@pytest.mark.parametrize("case", CASES, ids=[c[0] + ("-sq" if c[1].get("smooth_q") else "") for c in CASES])
def test_full_size_sampled_parity(case):
    name, over, (b, h), fwd_sel, q_sel, kv_sel = case
    w = workloads.get(name, **over)
    x = workloads.make_inputs(w, seed=0)
    q, O, L, dQ, dK, dV = _run_gpu(w, x)
    T = w.N // 64
    q_blocks = sorted({i % T for i in q_sel})
    kv_blocks = sorted({j % T for j in kv_sel})

    prep = osage.prepare(x["Q"], x["K"], x["V"], smooth_q=w.smooth_q)
    for k in ("Qh", "Kh", "Vh"):
        assert np.array_equal(getattr(q, k).cpu().numpy(), prep[k]), k
    for k in ("sQ", "sK", "sV", "muK") + (("muQ",) if w.smooth_q else ()):
        assert np.array_equal(getattr(q, k).cpu().numpy().view(np.uint32), np.asarray(prep[k], np.float32).view(np.uint32)), k

    # oracle forward on the rows the sampled tiles need
    if fwd_sel is None:
        fwd_blocks = None
    else:
        need = set(q_blocks)
        for j in kv_blocks:                          # causal: dK/dV of key block j sees query blocks >= j
            need.update(range(j, T))
        fwd_blocks = sorted(need)
    Oref, Lref = osage.sage_forward(prep, w.causal, q_blocks=fwd_blocks, heads=[(b, h)])
    rows = np.concatenate([np.arange(64 * i, 64 * i + 64) for i in (range(T) if fwd_blocks is None else fwd_blocks)])
    O_stored = workloads.round_to(Oref.astype(np.float32), w.dtype)
    L_stored = Lref.astype(np.float32)
    Og = O.float().cpu().numpy()[b, h]
    assert rel_l2(Og[rows], O_stored[b, h][rows]) <= 1e-3, rel_l2(Og[rows], O_stored[b, h][rows])
    Lg = L.cpu().numpy()[b, h]
    assert np.max(np.abs(Lg[rows] - L_stored[b, h][rows])) <= 1e-3 * max(1.0, float(np.max(np.abs(L_stored[b, h][rows]))))

    # oracle backward on the sampled dQ rows and dK / dV rows
    prep["V16"] = np.asarray(x["V"], np.float64)
    g = osage.sage_backward(prep, O_stored, L_stored, x["dO"], w.causal, q_blocks=q_blocks,
                            kv_blocks=kv_blocks, heads=[(b, h)])
    qrows = np.concatenate([np.arange(64 * i, 64 * i + 64) for i in q_blocks])
    krows = np.concatenate([np.arange(64 * j, 64 * j + 64) for j in kv_blocks])
    for nm, got, want, r in (("dQ", dQ, g["dQ"], qrows), ("dK", dK, g["dK"], krows), ("dV", dV, g["dV"], krows)):
        gv = got.cpu().numpy()[b, h][r]
        assert np.all(np.isfinite(gv)), nm
        err = rel_l2(gv, want[b, h][r])
        assert err <= 1e-3, (nm, err)


def test_full_size_fp8_headline():
    """The FP8 variant on the headline workload: E4M3 codes and scales byte for byte, sampled
    rows of head (0, 9) within rel-l2 1e-3 of the oracle's FP8 arithmetic."""
    import bit_trainable_attention_sage_gb300 as sg
    from oracle import quant
    w = workloads.get("headline")
    x = workloads.make_inputs(w, seed=1)
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    q = sg.sage_quantize_smooth(Q, K, V, fp8=True)
    O, L = sg.sage_attn_fwd(q, causal=False)
    dQ, dK, dV = sg.sage_attn_bwd(q, V, O, L, dO, causal=False)
    assert sg.sage_device_status() == 0
    ar = osage.QUANTISED_FP8
    prep = osage.prepare(x["Q"], x["K"], x["V"], arith=ar)
    for k in ("Qh", "Kh", "Vh"):
        assert np.array_equal(getattr(q, k).cpu().numpy().view(np.uint8), quant.e4m3_encode(prep[k])), k
    for k in ("sQ", "sK", "sV"):
        assert np.array_equal(getattr(q, k).cpu().numpy().view(np.uint32), prep[k].view(np.uint32)), k
    b, h = 0, 9
    Oref, Lref = osage.sage_forward(prep, False, arith=ar, heads=[(b, h)])
    O_stored = workloads.round_to(Oref.astype(np.float32), w.dtype)
    assert rel_l2(O.float().cpu().numpy()[b, h], O_stored[b, h]) <= 1e-3
    prep["V16"] = np.asarray(x["V"], np.float64)
    g = osage.sage_backward(prep, O_stored, Lref.astype(np.float32), x["dO"], False, arith=ar,
                            q_blocks=[3, 120], kv_blocks=[0, 64], heads=[(b, h)])
    qrows = np.r_[192:256, 7680:7744]
    krows = np.r_[0:64, 4096:4160]
    for nm, got, want, r in (("dQ", dQ, g["dQ"], qrows), ("dK", dK, g["dK"], krows), ("dV", dV, g["dV"], krows)):
        err = rel_l2(got.cpu().numpy()[b, h][r], want[b, h][r])
        assert err <= 1e-3, (nm, err)


def test_full_size_fp4_headline():
    """The FP4 inference forward on the headline workload: NVFP4 codes and scales of the whole
    tensors as values, O and L of head (1, 2) within rel-l2 1e-3 of the oracle's FP4 forward."""
    import bit_trainable_attention_sage_gb300 as sg
    from oracle import fp4, quant
    w = workloads.get("headline")
    x = workloads.make_inputs(w, seed=2)
    Q, K, V = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V"))
    q = sg.sage_quantize_fp4(Q, K, V)
    O, L = sg.sage_attn_fwd_fp4(q, causal=False)
    assert sg.sage_device_status() == 0
    prep = fp4.quantize_fp4(x["Q"], x["K"], x["V"])
    for nm in ("Q", "K", "V"):
        c = getattr(q, nm + "c").cpu().numpy()
        vals = fp4.e2m1_decode(np.stack([c & 15, c >> 4], axis=-1).reshape(*c.shape[:-1], c.shape[-1] * 2))
        assert np.array_equal(vals, prep[nm + "c"]), nm
        assert np.array_equal(quant.e4m3_decode(getattr(q, "s" + nm).cpu().numpy()), prep["s" + nm]), nm
    b, h = 1, 2
    Oref, Lref = fp4.sage_fp4_forward(prep, False, heads=[(b, h)])
    O_stored = workloads.round_to(Oref.astype(np.float32), w.dtype)
    assert rel_l2(O.float().cpu().numpy()[b, h], O_stored[b, h]) <= 1e-3
    assert np.max(np.abs(L.cpu().numpy()[b, h] - Lref[b, h])) <= 1e-3 * max(1.0, float(np.max(np.abs(Lref[b, h]))))


@pytest.mark.parametrize("name,head,fwd_sel,q_sel,kv_sel", [
    ("headline", (1, 7), None, [2, 101], [0, 127]),
    ("longseq", (0, 5), "ends", [0, 1, -1], [-1, -2]),
], ids=["headline", "longseq"])
def test_full_size_qat(name, head, fwd_sel, q_sel, kv_sel):
    """Attn-QAT at full size, in the benchmark's launch configuration: the sampled head's
    fake-quantised Q', K', V' bit for bit, its forward R on the rows computed, O, O' and L on those
    rows, and dQ, dK, dV on the sampled blocks within rel-l2 1e-3 of the oracle."""
    import bit_trainable_attention_sage_gb300 as sg
    from oracle import qat as oqat
    w = workloads.get(name)
    x = workloads.make_inputs(w, seed=2)
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    Qf, Kf, Vf = sg.sage_qat_quantize(Q, K, V)
    O, Op, L, R = sg.sage_qat_fwd(Qf, Kf, Vf, causal=w.causal)
    dQ, dK, dV = sg.sage_qat_bwd(Qf, Kf, Vf, Op, L, R, dO, causal=w.causal)
    assert sg.sage_device_status() == 0
    b, h = head
    T = w.N // 64
    q_blocks = sorted({i % T for i in q_sel})
    kv_blocks = sorted({j % T for j in kv_sel})
    one = lambda k: np.ascontiguousarray(x[k][b:b + 1, h:h + 1])
    fq = oqat.fake_quant(one("Q"), one("K"), one("V"))
    for k, t in (("Qf", Qf), ("Kf", Kf), ("Vf", Vf)):
        assert np.array_equal(t[b, h].float().cpu().numpy(), fq[k][0, 0].astype(np.float32)), k
    if fwd_sel is None:
        fwd_blocks = None
    else:
        need = set(q_blocks)
        for j in kv_blocks:
            need.update(range(j, T))
        fwd_blocks = sorted(need)
    rnd = lambda a: workloads.round_to(a, w.dtype)
    Oref, Opref, Lref, Rref = oqat.qat_forward(fq, w.causal, rnd, q_blocks=fwd_blocks)
    rows = np.concatenate([np.arange(64 * i, 64 * i + 64) for i in (range(T) if fwd_blocks is None else fwd_blocks)])
    assert rel_l2(O[b, h].float().cpu().numpy()[rows], rnd(Oref[0, 0].astype(np.float32))[rows]) <= 1e-3
    assert rel_l2(Op[b, h].cpu().numpy()[rows], Opref[0, 0][rows]) <= 1e-3
    Lg = L[b, h].cpu().numpy()[rows]
    assert np.max(np.abs(Lg - Lref[0, 0][rows])) <= 1e-3 * max(1.0, float(np.max(np.abs(Lref[0, 0][rows]))))
    Rg = R[b, h].cpu().numpy()[:, rows]
    Rr = Rref[0, 0][:, rows]
    fin = np.isfinite(Rr)
    assert np.array_equal(np.isneginf(Rg[~np.isnan(Rr)]), np.isneginf(Rr[~np.isnan(Rr)]))
    assert np.max(np.abs(Rg[fin] - Rr[fin]) / np.maximum(1.0, np.abs(Rr[fin]))) < 1e-5
    g = oqat.qat_backward(fq, Opref.astype(np.float32), Lref.astype(np.float32), Rref, one("dO"), w.causal, rnd,
                          q_blocks=q_blocks, kv_blocks=kv_blocks)
    qrows = np.concatenate([np.arange(64 * i, 64 * i + 64) for i in q_blocks])
    krows = np.concatenate([np.arange(64 * j, 64 * j + 64) for j in kv_blocks])
    for nm, got, want, r in (("dQ", dQ, g["dQ"], qrows), ("dK", dK, g["dK"], krows), ("dV", dV, g["dV"], krows)):
        gv = got[b, h].cpu().numpy()[r]
        assert np.all(np.isfinite(gv)), nm
        err = rel_l2(gv, want[0, 0][r])
        assert err <= 1e-3, (nm, err)
