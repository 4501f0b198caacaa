"""GPU parity of the INT8-dP ablation (SAGE_FLAG_DP_INT8) against the oracle's same variant.

"SageAttention3 ..." (review), Table 1c compares keeping dP = dO V^T in 16 bits with forming it from
the INT8 codes of dO and V.  With the flag the backward kernel feeds the dP MMA the integer-valued
fp16 codes and scales the exact integer product by fl32(s_dO s_V).  dQ, dK, dV must match the
oracle's variant within rel-l2 1e-3, and must differ from the method's 16-bit-dP results by about
as much as the oracle's two variants differ.
"""
import numpy as np
import pytest

from tests.gpu_common import gpu_run, make_case, oracle_run, rel_l2

pytestmark = pytest.mark.gpu

CASES = [
    (256, 128, "fp16", False, {}),
    (320, 64, "bf16", True, {}),
    (192, 128, "fp16", True, dict(smooth_q=True)),
]


@pytest.mark.parametrize("case", CASES, ids=[f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}" for c in CASES])
def test_dp_int8_parity(case):
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    g8 = gpu_run(w, x, dp_int8=True)
    g16 = gpu_run(w, x)
    ref8 = oracle_run(w, x, record=False, dp_int8=True)
    ref16 = oracle_run(w, x, record=False)
    for k in ("dQ", "dK", "dV"):
        assert np.all(np.isfinite(g8[k])), k
        assert rel_l2(g8[k], ref8[k]) <= 1e-3, (k, rel_l2(g8[k], ref8[k]))
    # the flag takes effect: dQ moves away from the 16-bit-dP result as far as the oracle's does
    want = rel_l2(ref8["dQ"], ref16["dQ"])
    got = rel_l2(g8["dQ"], g16["dQ"])
    assert want > 1e-3
    assert 0.5 * want <= got <= 2.0 * want, (got, want)
