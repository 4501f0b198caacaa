"""The autograd wrapper: gradients equal the direct C calls' (dQ up to the order of its float32
reductions) and approximate full-precision attention's (the quantisation error of SageBwd,
cos > 0.99 on unit-variance inputs)."""
import numpy as np
import pytest
import torch

from tests.gpu_common import make_case, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal,dtype", [(False, "fp16"), (True, "bf16")])
def test_autograd_matches_direct_calls_and_fpa(causal, dtype):
    import bit_trainable_attention_sage_gb300 as sg
    w, x = make_case(256, 128, dtype, causal)
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    Qr, Kr, Vr = (t.clone().requires_grad_(True) for t in (Q, K, V))
    O = sg.sage_attention(Qr, Kr, Vr, causal=causal)
    O.backward(dO)
    # the same calls by hand
    q = sg.sage_quantize_smooth(Q, K, V)
    O2, L2 = sg.sage_attn_fwd(q, causal=causal)
    dQ, dK, dV = sg.sage_attn_bwd(q, V, O2, L2, dO, causal=causal)
    assert sg.sage_device_status() == 0
    assert torch.equal(O, O2)
    # dK and dV are deterministic; dQ is summed with float32 reductions in any order
    for g, ref in ((Kr.grad, dK), (Vr.grad, dV)):
        assert g.dtype == Q.dtype
        assert torch.equal(g, ref.to(Q.dtype))
    assert rel_l2(Qr.grad.float().cpu().numpy(), dQ.to(Q.dtype).float().cpu().numpy()) <= 1e-3
    # full-precision attention in float32 with torch's own autograd
    Qf, Kf, Vf = (t.float().clone().requires_grad_(True) for t in (Q, K, V))
    S = Qf @ Kf.transpose(-1, -2) / np.sqrt(w.d)
    if causal:
        S = S.masked_fill(torch.ones(w.N, w.N, dtype=torch.bool, device=S.device).triu(1), float("-inf"))
    Of = torch.softmax(S, -1) @ Vf
    Of.backward(dO.float())
    for got, ref in ((O, Of), (Qr.grad, Qf.grad), (Kr.grad, Kf.grad), (Vr.grad, Vf.grad)):
        a, b = got.detach().float().flatten(), ref.detach().float().flatten()
        cos = float(torch.dot(a, b) / (a.norm() * b.norm()))
        assert cos > 0.99, cos


@pytest.mark.parametrize("causal,dtype", [(False, "bf16"), (True, "fp16")])
def test_qat_autograd_matches_direct_calls(causal, dtype):
    """sage_attention_qat: the output and the gradients (cast to the input dtype) are those of the
    three Attn-QAT calls (dQ up to the order of its float32 reductions), and the QAT output is
    an approximation of full-precision attention (cos > 0.98 at 4 bits)."""
    import bit_trainable_attention_sage_gb300 as sg
    w, x = make_case(256, 64, dtype, causal)
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    Qr, Kr, Vr = (t.clone().requires_grad_(True) for t in (Q, K, V))
    O = sg.sage_attention_qat(Qr, Kr, Vr, causal=causal)
    O.backward(dO)
    Qf, Kf, Vf = sg.sage_qat_quantize(Q, K, V)
    O2, Op, L, R = sg.sage_qat_fwd(Qf, Kf, Vf, causal=causal)
    dQ, dK, dV = sg.sage_qat_bwd(Qf, Kf, Vf, Op, L, R, dO, causal=causal)
    assert sg.sage_device_status() == 0
    assert torch.equal(O, O2)
    for g, ref in ((Kr.grad, dK), (Vr.grad, dV)):
        assert g.dtype == Q.dtype and torch.equal(g, ref.to(Q.dtype))
    assert rel_l2(Qr.grad.float().cpu().numpy(), dQ.to(Q.dtype).float().cpu().numpy()) <= 1e-3
    S = Q.float() @ K.float().transpose(-1, -2) / np.sqrt(w.d)
    if causal:
        S = S.masked_fill(torch.ones(w.N, w.N, dtype=torch.bool, device=S.device).triu(1), float("-inf"))
    Ofp = torch.softmax(S, -1) @ V.float()
    cos = torch.nn.functional.cosine_similarity(O.float().flatten(), Ofp.flatten(), dim=0).item()
    assert cos > 0.98, cos
