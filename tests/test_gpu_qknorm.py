"""GPU parity of the QK-norm prologue and its gradient ("SageBwd: A Trainable Low-bit Attention"
(structured summary), QK-norm: x / sqrt(mean x^2 + eps) * gamma, eps 1e-6) against the oracle.

The fused quantiser must give the oracle's row factors, normalised 16-bit tensors, codes, scales
and means bit for bit; the whole path (fused quantise -> forward -> backward -> norm gradient)
must match the oracle's chain within rel-l2 1e-3; the norm gradient kernel alone (float32
arithmetic) within rel-l2 1e-5 of the float64 oracle.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import qknorm, quant
from oracle import sage as osage
from tests.gpu_common import rel_l2, to_dev

pytestmark = pytest.mark.gpu

EPS = np.float32(1e-6)


def _raw(N, d, dtype, seed, B=1, H=2):
    """Un-normalised Q, K (per-token scales spread over two decades, a K channel offset), V, dO."""
    rng = np.random.default_rng(seed)
    rnd = lambda a: workloads.round_to(a.astype(np.float32), dtype)
    tok = lambda: np.exp(rng.normal(0.0, 1.2, (B, H, N, 1)))
    Q = rnd(rng.standard_normal((B, H, N, d)) * tok())
    K = rnd((rng.standard_normal((B, H, N, d)) + rng.normal(0, 2.0, (B, H, 1, d))) * tok())
    V = rnd(rng.standard_normal((B, H, N, d)))
    dO = rnd(rng.standard_normal((B, H, N, d)) * 1e-2)
    g = rng.uniform(0.5, 1.5, (2, d)).astype(np.float32)
    return Q, K, V, dO, g


def _oracle_prologue(Q, K, gq, gk, dtype):
    rnd = lambda a: workloads.round_to(a, dtype)
    Yq, rq = qknorm.rms_norm(Q, gq, EPS, rnd)
    Yk, rk = qknorm.rms_norm(K, gk, EPS, rnd)
    return Yq, rq, Yk, rk


def _bits(t):
    return t.cpu().numpy().view(np.uint32) if t.dtype == torch.float32 else t.cpu().view(torch.int16).numpy()


PRO_CASES = [
    (256, 128, "fp16", True, False),
    (192, 64, "bf16", True, True),
    (128, 128, "bf16", False, False),
    (320, 64, "fp16", False, True),
]


@pytest.mark.parametrize("case", PRO_CASES, ids=[f"N{c[0]}-d{c[1]}-{c[2]}-{'g' if c[3] else 'nog'}-{'sq' if c[4] else 'nosq'}" for c in PRO_CASES])
def test_qknorm_prologue_bit_exact(case):
    import bit_trainable_attention_sage_gb300 as sg
    N, d, dtype, with_g, smooth_q = case
    Q, K, V, _, g = _raw(N, d, dtype, seed=N + d)
    gq, gk = (g[0], g[1]) if with_g else (None, None)
    dev = lambda a: to_dev(a, dtype)
    gdev = lambda a: None if a is None else torch.from_numpy(a).cuda()
    q = sg.sage_quantize_smooth_qknorm(dev(Q), dev(K), dev(V), gamma_q=gdev(gq), gamma_k=gdev(gk),
                                       eps=float(EPS), smooth_q=smooth_q, keep_normed=True)
    torch.cuda.synchronize()
    Yq, rq, Yk, rk = _oracle_prologue(Q, K, gq, gk, dtype)
    assert np.array_equal(q.rQ.cpu().numpy().view(np.uint32), rq.view(np.uint32))
    assert np.array_equal(q.rK.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(q.Qn.float().cpu().numpy(), Yq)
    assert np.array_equal(q.Kn.float().cpu().numpy(), Yk)
    prep = quant.quantize_smooth(Yq, Yk, V, smooth_q=smooth_q)
    for k in ("Qh", "Kh", "Vh"):
        assert np.array_equal(getattr(q, k).cpu().numpy(), prep[k]), k
    for k in ("sQ", "sK", "sV", "muK") + (("muQ",) if smooth_q else ()):
        assert np.array_equal(getattr(q, k).cpu().numpy().view(np.uint32), np.asarray(prep[k], np.float32).view(np.uint32)), k


PATH_CASES = [
    (256, 128, "bf16", True, False, False),
    (192, 64, "fp16", False, True, False),
    (256, 128, "fp16", True, False, True),
]


@pytest.mark.parametrize("case", PATH_CASES, ids=[f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}-{'sq' if c[4] else 'nosq'}-{'fp8' if c[5] else 'int8'}" for c in PATH_CASES])
def test_qknorm_path_parity(case):
    """sage_attention(qk_norm=True) forward and backward (including the gammas' gradients) against
    the oracle chain: norm -> SageBwd -> norm gradient."""
    import bit_trainable_attention_sage_gb300 as sg
    N, d, dtype, causal, smooth_q, fp8 = case
    Q, K, V, dO, g = _raw(N, d, dtype, seed=7 * N + d)
    dev = lambda a: to_dev(a, dtype).requires_grad_(True)
    Qd, Kd, Vd = dev(Q), dev(K), dev(V)
    gq = torch.from_numpy(g[0]).cuda().requires_grad_(True)
    gk = torch.from_numpy(g[1]).cuda().requires_grad_(True)
    O = sg.sage_attention(Qd, Kd, Vd, causal=causal, smooth_q=smooth_q, fp8=fp8, qk_norm=True,
                          gamma_q=gq, gamma_k=gk, eps=float(EPS))
    O.backward(to_dev(dO, dtype))
    assert sg.sage_device_status() == 0
    Yq, rq, Yk, rk = _oracle_prologue(Q, K, g[0], g[1], dtype)
    ref = osage.run(Yq, Yk, V, dO, causal, lambda a: workloads.round_to(a, dtype), smooth_q=smooth_q,
                    arith=osage.QUANTISED_FP8 if fp8 else osage.QUANTISED)
    dQ, dgq = qknorm.rms_norm_bwd(Q, g[0], rq, ref["dQ"])
    dK, dgk = qknorm.rms_norm_bwd(K, g[1], rk, ref["dK"])
    assert rel_l2(O.detach().float().cpu().numpy(), ref["O_stored"]) <= 1e-3
    # the gradients come back in the 16-bit input dtype: the bar is 1e-3 beyond that rounding
    for name, got, want in (("dQ", Qd.grad, dQ), ("dK", Kd.grad, dK), ("dV", Vd.grad, ref["dV"])):
        own = rel_l2(workloads.round_to(want.astype(np.float32), dtype), want)
        err = rel_l2(got.float().cpu().numpy(), want)
        assert err <= 1e-3 + own, (name, err, own)
    for name, got, want in (("dgamma_q", gq.grad, dgq), ("dgamma_k", gk.grad, dgk)):
        assert rel_l2(got.cpu().numpy(), want) <= 1e-3, (name, rel_l2(got.cpu().numpy(), want))


@pytest.mark.parametrize("dtype,d,with_g", [("fp16", 128, True), ("bf16", 64, False)])
def test_qknorm_bwd_kernel(dtype, d, with_g):
    import bit_trainable_attention_sage_gb300 as sg
    N = 512
    Q, K, V, _, g = _raw(N, d, dtype, seed=99, B=2, H=3)
    gq = g[0] if with_g else None
    rng = np.random.default_rng(5)
    dY = rng.standard_normal(Q.shape).astype(np.float32)
    gdev = None if gq is None else torch.from_numpy(gq).cuda()
    q = sg.sage_quantize_smooth_qknorm(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype), gamma_q=gdev,
                                       eps=float(EPS))
    dX, dg = sg.sage_qknorm_bwd(to_dev(Q, dtype), q.rQ, torch.from_numpy(dY).cuda(), gamma=gdev)
    torch.cuda.synchronize()
    _, rq = qknorm.rms_norm(Q, gq, EPS, lambda a: workloads.round_to(a, dtype))
    want_dx, want_dg = qknorm.rms_norm_bwd(Q, gq, rq, dY)
    assert rel_l2(dX.cpu().numpy(), want_dx) <= 1e-5
    assert rel_l2(dg.cpu().numpy(), want_dg) <= 1e-5
    # without dgamma the call writes dX alone
    dX2, dg2 = sg.sage_qknorm_bwd(to_dev(Q, dtype), q.rQ, torch.from_numpy(dY).cuda(), gamma=gdev, want_dgamma=False)
    assert dg2 is None and torch.equal(dX, dX2)


def test_qknorm_refuses_bad_eps():
    import bit_trainable_attention_sage_gb300 as sg
    Q, K, V, _, _ = _raw(128, 64, "fp16", seed=1)
    with pytest.raises(sg.SageError):
        sg.sage_quantize_smooth_qknorm(to_dev(Q, "fp16"), to_dev(K, "fp16"), to_dev(V, "fp16"), eps=-1.0)


@pytest.mark.parametrize("dtype,d", [("fp16", 128), ("bf16", 64)])
def test_qknorm_row_factor_many_rows(dtype, d):
    """The row factor is the float32 nearest to 1 / sqrt(mean x^2 + eps) on every one of 2 x 32768
    rows whose per-token scales span four decades (the kernel's float32 candidate is corrected from
    its residual, with a float64 decision near rounding boundaries); the normalised tensors, codes,
    scales and means that follow stay bit-exact."""
    import bit_trainable_attention_sage_gb300 as sg
    B, H, N = 1, 8, 4096
    rng = np.random.default_rng(17)
    rnd = lambda a: workloads.round_to(a.astype(np.float32), dtype)
    tok = lambda: np.exp(rng.normal(0.0, 2.0, (B, H, N, 1)))
    Q = rnd(rng.standard_normal((B, H, N, d)) * tok())
    K = rnd(rng.standard_normal((B, H, N, d)) * tok())
    V = rnd(rng.standard_normal((B, H, N, d)))
    q = sg.sage_quantize_smooth_qknorm(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype), eps=float(EPS),
                                       keep_normed=True)
    torch.cuda.synchronize()
    Yq, rq, Yk, rk = _oracle_prologue(Q, K, None, None, dtype)
    for name, got, want in (("rQ", q.rQ, rq), ("rK", q.rK, rk)):
        g = got.cpu().numpy()
        ulps = np.abs(g.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
        print(f"\n{name}: {int((ulps != 0).sum())} of {ulps.size} rows differ, largest {int(ulps.max())} ulp")
        assert ulps.max() <= 1, name
        assert np.array_equal(g.view(np.uint32), want.view(np.uint32)), name
    assert np.array_equal(q.Qn.float().cpu().numpy(), Yq)
    assert np.array_equal(q.Kn.float().cpu().numpy(), Yk)
    prep = quant.quantize_smooth(Yq, Yk, V)
    for k in ("Qh", "Kh", "Vh"):
        assert np.array_equal(getattr(q, k).cpu().numpy(), prep[k]), k
    for k in ("sQ", "sK", "muK"):
        assert np.array_equal(getattr(q, k).cpu().numpy().view(np.uint32), np.asarray(prep[k], np.float32).view(np.uint32)), k
