"""GPU parity of the Attn-QAT path against the oracle ("Attn-QAT: 4-Bit Attention With
Quantization-Aware Training", technical summary, sections 2.1-2.3).

Bit-exact: the fake-quantised Q', K', V' (NVFP4 values in the input type).  R, the forward's
row maxima, to float32 accuracy (the products are summed in the tensor core's float32
accumulator; the oracle's are exact) and -inf exactly where a row sees no key of the block.
O, O', dQ, dK, dV within rel-l2 1e-3 of the oracle run on the same inputs: the kernels' ex2 is
the hardware approximation and their sums are float32, which can move an FP4 code of P across a
rounding boundary now and then.  Property: without the high-precision O' (D from O) the
gradients would differ far more than the tolerance -- the kernel's D is checked against D from
its own O' and O.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import qat
from tests.gpu_common import make_case, rel_l2, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    (128, 64, "fp16", False),
    (320, 128, "fp16", True),        # ragged tail of the 128-key tile, causal
    (256, 128, "bf16", False),
    (192, 64, "bf16", True),
    (64, 128, "fp16", True),         # a single block: the diagonal only
    (384, 64, "fp16", False),
]
IDS = [f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}" for c in CASES]


def _gpu(x, dtype, causal):
    import bit_trainable_attention_sage_gb300 as sg
    Q, K, V, dO = (to_dev(x[k], dtype) for k in ("Q", "K", "V", "dO"))
    Qf, Kf, Vf = sg.sage_qat_quantize(Q, K, V)
    O, Op, L, R = sg.sage_qat_fwd(Qf, Kf, Vf, causal=causal)
    dQ, dK, dV = sg.sage_qat_bwd(Qf, Kf, Vf, Op, L, R, dO, causal=causal)
    st = sg.sage_device_status()
    assert st == 0, sg.sage_status_string(st)
    f = lambda t: t.float().cpu().numpy()
    return dict(Qf=f(Qf), Kf=f(Kf), Vf=f(Vf), O=f(O), Op=f(Op), L=f(L), R=f(R), dQ=f(dQ), dK=f(dK), dV=f(dV))


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_qat_parity(case):
    N, d, dtype, causal = case
    w, x = make_case(N, d, dtype, causal)
    g = _gpu(x, dtype, causal)
    ref = qat.run(x["Q"], x["K"], x["V"], x["dO"], causal, lambda a: workloads.round_to(a, dtype))
    for k in ("Qf", "Kf", "Vf"):
        assert np.array_equal(g[k], ref["fq"][k].astype(np.float32)), k
    # R where the oracle's forward visits the pair
    Rr = ref["R"]
    seen = ~np.isnan(Rr)
    fin = seen & np.isfinite(Rr)
    assert np.array_equal(np.isneginf(g["R"][seen]), np.isneginf(Rr[seen]))
    assert np.max(np.abs(g["R"][fin] - Rr[fin]) / np.maximum(1.0, np.abs(Rr[fin]))) < 1e-5
    assert rel_l2(g["O"], ref["O_stored"]) <= 1e-3, rel_l2(g["O"], ref["O_stored"])
    assert rel_l2(g["Op"], ref["Op"]) <= 1e-3, rel_l2(g["Op"], ref["Op"])
    assert np.max(np.abs(g["L"] - ref["L"])) <= 1e-3 * max(1.0, np.max(np.abs(ref["L"])))
    for k in ("dQ", "dK", "dV"):
        assert np.all(np.isfinite(g[k])), k
        assert rel_l2(g[k], ref[k]) <= 1e-3, (k, rel_l2(g[k], ref[k]))


def test_qat_refuses_smoothing_and_flags():
    import ctypes
    import bit_trainable_attention_sage_gb300 as sg
    w, x = make_case(128, 64, "fp16", False)
    Q, K, V = (to_dev(x[k], "fp16") for k in ("Q", "K", "V"))
    Qf, Kf, Vf = (torch.empty_like(t) for t in (Q, K, V))
    p = sg.make_params(1, 2, 128, 64, 0, False)                   # smooth_k = 1
    st = sg.lib().sage_qat_quantize(ctypes.byref(p), Q.data_ptr(), K.data_ptr(), V.data_ptr(), Qf.data_ptr(),
                                    Kf.data_ptr(), Vf.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 2
