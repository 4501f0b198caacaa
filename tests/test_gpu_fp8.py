"""GPU parity of the FP8 SageBwd variant (SAGE_FLAG_FP8) against the oracle's FP8 arithmetic.

"SageAttention3 ..." (review), INT8 vs FP8 training: the same SageBwd with E4M3 codes.  The
quantiser's E4M3 codes and block scales must be bit-exact; O, L, dQ, dK, dV within rel-l2 1e-3 of
the oracle's FP8 run (the block products of E4M3 values are exact in float64 but summed in the
tensor core's float32 accumulator, which moves a P or dS code across a rounding boundary now and
then); and the flag must move the results away from the INT8 ones by about as much as it moves
the oracle's.
"""
import numpy as np
import pytest
import torch

from oracle import quant
from tests.gpu_common import gpu_run, make_case, oracle_run, rel_l2, to_dev

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


def _codes_match(gpu_codes, oracle_values):
    """GPU E4M3 bit patterns against the oracle's code values, byte for byte."""
    return np.array_equal(gpu_codes.view(np.uint8), quant.e4m3_encode(oracle_values))


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fp8_parity(case):
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    g8 = gpu_run(w, x, fp8=True)
    ref = oracle_run(w, x, record=False, fp8=True)
    prep = ref["prep"]
    for k in ("Qh", "Kh", "Vh"):
        assert _codes_match(g8["q"][k], prep[k]), k
    for k in ("sQ", "sK", "sV", "muK"):
        assert np.array_equal(g8["q"][k].view(np.uint32), np.asarray(prep[k], np.float32).view(np.uint32)), k
    assert rel_l2(g8["O"], ref["O_stored"]) <= 1e-3, rel_l2(g8["O"], ref["O_stored"])
    assert np.max(np.abs(g8["L"] - ref["L_stored"])) <= 1e-3 * max(1.0, np.max(np.abs(ref["L_stored"])))
    for k in ("dQ", "dK", "dV"):
        assert np.all(np.isfinite(g8[k])), k
        assert rel_l2(g8[k], ref[k]) <= 1e-3, (k, rel_l2(g8[k], ref[k]))


def test_fp8_flag_takes_effect():
    w, x = make_case(256, 128, "fp16", False)
    g8, gi = gpu_run(w, x, fp8=True), gpu_run(w, x)
    r8, ri = oracle_run(w, x, record=False, fp8=True), oracle_run(w, x, record=False)
    for k in ("O", "dQ", "dK", "dV"):
        a, b = (g8[k], gi[k]) if k != "O" else (g8["O"], gi["O"])
        want = rel_l2(r8[k] if k != "O" else r8["O_stored"], ri[k] if k != "O" else ri["O_stored"])
        got = rel_l2(a, b)
        assert want > 1e-3, (k, want)
        assert 0.5 * want <= got <= 2.0 * want, (k, got, want)


def test_fp8_noalloc_quantiser_matches():
    import bit_trainable_attention_sage_gb300 as sg
    w, x = make_case(256, 64, "bf16", False, smooth_q=True)
    Q, K, V = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V"))
    a = sg.sage_quantize_smooth(Q, K, V, smooth_q=True, fp8=True)
    b = sg.sage_quantize_smooth_noalloc(Q, K, V, smooth_q=True, fp8=True)
    torch.cuda.synchronize()
    for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK", "muQ"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    assert a.fp8 and b.fp8


def test_fp8_refuses_dump_and_int8_dp():
    import bit_trainable_attention_sage_gb300 as sg
    w, x = make_case(128, 64, "fp16", False)
    Q, K, V, dO = (to_dev(x[k], w.dtype) for k in ("Q", "K", "V", "dO"))
    q = sg.sage_quantize_smooth(Q, K, V, fp8=True)
    O, L = sg.sage_attn_fwd(q, causal=False)
    with pytest.raises(sg.SageError):
        sg.sage_attn_bwd(q, V, O, L, dO, causal=False, dp_int8=True)
    buf = torch.zeros(sg.sage_dump_bytes(1, 2, 128, 64, 0), dtype=torch.uint8, device="cuda")
    with pytest.raises(sg.SageError):
        sg.sage_attn_fwd(q, causal=False, dump=buf)
