"""SAGE_FLAG_OPS16, the binding's default: the quantise call also writes each code's exact fp16
value (the tensor cores' operand), and the forward and backward calls read those copies instead of
widening the codes themselves.

Checked through the binding against the same calls without the flag, on the same codes: the
copies equal the codes' values (int8 codes, or E4M3 bit patterns with SAGE_FLAG_FP8); O and L are
bit-identical; dK and dV bit-identical; dQ, whose float32 reductions run in any order, within
rel-l2 1e-6.  Shapes: d = 64 and 128, fp16 and bf16, causal and not, Q-smoothing, FP8, the QK-norm
form and the allocation-free form of the quantise call.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests.gpu_common import make_case, rel_l2, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # N, d, dtype, causal, extra, quantise form
    (320, 128, "fp16", True, {}, "plain"),
    (384, 64, "bf16", True, dict(smooth_q=True), "plain"),
    (256, 128, "fp16", False, dict(fp8=True), "plain"),
    (256, 128, "bf16", False, dict(qk="qknorm"), "qknorm"),
    (192, 64, "fp16", False, {}, "noalloc"),
]


def _values(codes: torch.Tensor, fp8: bool) -> torch.Tensor:
    if fp8:
        return codes.view(torch.float8_e4m3fn).to(torch.float16)
    return codes.to(torch.float16)


@pytest.mark.parametrize("case", CASES, ids=[f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}-{c[5]}-"
                                              + "-".join(f"{k}={v}" for k, v in c[4].items()) for c in CASES])
def test_operand_copies_match_widened_path(case):
    import bit_trainable_attention_sage_gb300 as sg
    N, d, dtype, causal, extra, form = case
    fp8 = extra.pop("fp8", False) if "fp8" in extra else False
    w, x = make_case(N, d, dtype, causal, B=2, H=2, **extra)
    Q, K, V, dO = (to_dev(x[k], dtype) for k in ("Q", "K", "V", "dO"))
    if form == "qknorm":
        q = sg.sage_quantize_smooth_qknorm(Q, K, V, smooth_q=w.smooth_q)
    elif form == "noalloc":
        q = sg.sage_quantize_smooth_noalloc(Q, K, V, smooth_q=w.smooth_q)
    else:
        q = sg.sage_quantize_smooth(Q, K, V, smooth_q=w.smooth_q, fp8=fp8)
    assert q.ops16 is not None
    for i, name in enumerate(("Qh", "Kh", "Vh")):
        assert torch.equal(q.ops16[i], _values(getattr(q, name), fp8)), name
    plain = dataclasses.replace(q, ops16=None)
    Kb = (q.Kn if form == "qknorm" else K) if w.smooth_q else None
    O1, L1 = sg.sage_attn_fwd(q, causal=causal, K=Kb)
    O0, L0 = sg.sage_attn_fwd(plain, causal=causal, K=Kb)
    assert torch.equal(O1, O0) and torch.equal(L1, L0)
    g1 = sg.sage_attn_bwd(q, V, O1, L1, dO, causal=causal, K=Kb)
    g0 = sg.sage_attn_bwd(plain, V, O0, L0, dO, causal=causal, K=Kb)
    assert sg.sage_device_status() == 0
    assert torch.equal(g1[1], g0[1]) and torch.equal(g1[2], g0[2])
    assert rel_l2(g1[0].cpu().numpy(), g0[0].cpu().numpy()) <= 1e-6
    assert np.all(np.isfinite(g1[0].cpu().numpy()))
