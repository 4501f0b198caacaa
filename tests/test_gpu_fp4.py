"""GPU parity of the SageAttention3 FP4 inference forward against the oracle ("SageAttention3 ..."
(review), eq. (2)-(6): NVFP4 E2M1 codes with E4M3 scales per 1 x 16 block, two-level P).

The quantiser's codes and scales must be bit-exact (compared as values; the sign of a zero code
is not compared); O and L within rel-l2 1e-3 of the oracle's FP4 forward: the dequantised block
products are exact in float64 on the oracle's side but summed in the tensor core's float32
accumulator, which can move a P code across a rounding boundary now and then.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import fp4, quant
from tests.gpu_common import make_case, rel_l2, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    (256, 128, "fp16", False, {}),
    (320, 64, "bf16", True, {}),
    (192, 128, "fp16", True, dict(smooth_q=True)),
    (64, 64, "fp16", False, {}),
    (384, 128, "bf16", False, dict(qk="qknorm", k_offset_var=4.0)),
]
IDS = [f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}" + ("-sq" if c[4].get("smooth_q") else "")
       + ("-qknorm" if c[4].get("qk") else "") for c in CASES]


def _nibbles(codes):
    """(..., d/2) packed bytes -> (..., d) E2M1 values, the even element from the low nibble."""
    c = codes.cpu().numpy()
    lo, hi = c & 15, c >> 4
    return fp4.e2m1_decode(np.stack([lo, hi], axis=-1).reshape(*c.shape[:-1], c.shape[-1] * 2))


def _scales(s):
    return quant.e4m3_decode(s.cpu().numpy())


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fp4_forward_parity(case):
    import bit_trainable_attention_sage_gb300 as sg
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    Q, K, V = (to_dev(x[k], dtype) for k in ("Q", "K", "V"))
    q = sg.sage_quantize_fp4(Q, K, V, smooth_q=w.smooth_q)
    O, L = sg.sage_attn_fwd_fp4(q, causal=causal, K=K if w.smooth_q else None)
    assert sg.sage_device_status() == 0
    prep = fp4.quantize_fp4(x["Q"], x["K"], x["V"], smooth_q=w.smooth_q)
    for name in ("Q", "K", "V"):
        assert np.array_equal(_nibbles(getattr(q, name + "c")), prep[name + "c"]), name
        assert np.array_equal(_scales(getattr(q, "s" + name)), prep["s" + name]), name
    assert np.array_equal(q.muK.cpu().numpy().view(np.uint32), prep["muK"].view(np.uint32))
    Oref, Lref = fp4.sage_fp4_forward(prep, causal)
    O_stored = workloads.round_to(Oref.astype(np.float32), dtype)
    err = rel_l2(O.float().cpu().numpy(), O_stored)
    assert err <= 1e-3, err
    assert np.max(np.abs(L.cpu().numpy() - Lref)) <= 1e-3 * max(1.0, np.max(np.abs(Lref)))


def test_fp4_refuses_flags():
    import bit_trainable_attention_sage_gb300 as sg
    w, x = make_case(128, 64, "fp16", False)
    Q, K, V = (to_dev(x[k], "fp16") for k in ("Q", "K", "V"))
    q = sg.sage_quantize_fp4(Q, K, V)
    L = sg.lib()
    import ctypes
    p = sg.make_params(1, 2, 128, 64, 0, False, fp8=True)
    O = torch.empty((1, 2, 128, 64), dtype=torch.float16, device="cuda")
    Lse = torch.empty((1, 2, 128), dtype=torch.float32, device="cuda")
    st = L.sage_attn_fwd_fp4(ctypes.byref(p), q.Qc.data_ptr(), q.Kc.data_ptr(), q.Vc.data_ptr(), q.sQ.data_ptr(),
                             q.sK.data_ptr(), q.sV.data_ptr(), None, None, None, O.data_ptr(), Lse.data_ptr(),
                             None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 2
