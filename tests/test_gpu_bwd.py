"""GPU parity of sage_attn_bwd against the CPU oracle.

Bit-exact: dO^ codes and block scales, the recomputed integer Q^ K^T products (debug dump).
P and dS codes: within one code of the oracle's on at most 2e-3 of the entries (float32 decisions
on both sides; the kernel's exp2 is the hardware approximation and its L and D carry the forward's
own float32 rounding).  dQ, dK, dV: rel-l2 <= 1e-3 against the oracle.  Property at any size: dV
equals the float64 sum of the kernel's own dumped codes times their scales.
"""
import numpy as np
import pytest

from tests.gpu_common import causal_mask_full, gpu_run, make_case, oracle_run, rel_l2, visited_blocks

pytestmark = pytest.mark.gpu

CASES = [
    (128, 64, "fp16", False, {}),
    (320, 128, "fp16", True, {}),
    (384, 64, "bf16", True, dict(smooth_q=True)),
    (512, 128, "bf16", False, dict(qk="qknorm", k_offset_var=4.0, do_var=1e-4)),
    (256, 128, "fp16", False, dict(sigma=5.0)),
    (192, 64, "fp16", True, dict(qk="outlier", smooth_q=True)),
    (64, 128, "fp16", True, {}),                      # one block: diagonal only
    (64, 64, "bf16", False, dict(smooth_q=True)),     # one block, Q-smoothing
]


def _ids(c):
    return f"N{c[0]}-d{c[1]}-{c[2]}-{'causal' if c[3] else 'full'}-{'-'.join(f'{k}={v}' for k, v in c[4].items())}"


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_backward_parity(case):
    N, d, dtype, causal, extra = case
    w, x = make_case(N, d, dtype, causal, **extra)
    g = gpu_run(w, x, dump=True)
    ref = oracle_run(w, x)
    for k in ("dQ", "dK", "dV"):
        assert np.all(np.isfinite(g[k])), k
        assert rel_l2(g[k], ref[k]) <= 1e-3, (k, rel_l2(g[k], ref[k]))
    dmp = g["dump"]
    assert np.array_equal(dmp["dOh"], ref["dOh"])
    assert np.array_equal(dmp["sdO"].view(np.uint32), ref["sdO"].view(np.uint32))
    # D is formed from the kernel's own stored O (its 16-bit rounding differs from the oracle's)
    D_own = (x["dO"].astype(np.float64) * g["O"].astype(np.float64)).sum(-1)
    assert rel_l2(dmp["D"], D_own) <= 1e-5
    assert rel_l2(dmp["D"], ref["D"]) <= 1e-3
    mask = causal_mask_full(N) if causal else np.zeros((N, N), bool)
    rec = ref["record"]
    prep = ref["prep"]
    n_codes = n_diff_p = n_diff_ds = 0
    for b in range(w.B):
        for h in range(w.H):
            # the backward records dequantised P and dS; recover codes with the oracle's scales
            for (i, j) in visited_blocks(N, causal):
                rows, cols = slice(64 * i, 64 * i + 64), slice(64 * j, 64 * j + 64)
                live = ~mask[rows, cols]
                S_ref = prep["Qh"][b, h, rows].astype(np.int64) @ prep["Kh"][b, h, cols].astype(np.int64).T
                assert np.array_equal(dmp["S"][b, h, rows, cols][live], S_ref[live]), (b, h, i, j)
                for name, key in (("P", "P"), ("dS", "dS")):
                    code = dmp[name][b, h, rows, cols].astype(np.int64)
                    deq = rec[(b, h)][key][rows, cols]
                    scale = np.abs(deq).max()
                    sgpu = dmp["sP" if name == "P" else "sdS"][b, h, i, j]
                    if scale == 0:
                        assert not code[live].any() and sgpu == 0
                        continue
                    ref_code = np.rint(deq / (scale / 127.0)).astype(np.int64)
                    diff = np.abs(code - ref_code)[live]
                    assert diff.max(initial=0) <= 1, (name, b, h, i, j)
                    assert abs(sgpu - scale / 127.0) <= 1e-3 * scale / 127.0, (name, b, h, i, j)
                    if name == "P":
                        n_diff_p += int((diff != 0).sum())
                    else:
                        n_diff_ds += int((diff != 0).sum())
                n_codes += int(live.sum())
    print(f"\n{_ids(case)}: P code flips {n_diff_p}/{n_codes}, dS code flips {n_diff_ds}/{n_codes}, "
          + ", ".join(f"{k} rel-l2 {rel_l2(g[k], ref[k]):.2e}" for k in ("dQ", "dK", "dV")))
    assert n_diff_p <= 2e-3 * n_codes, (n_diff_p, n_codes)
    assert n_diff_ds <= 2e-3 * n_codes, (n_diff_ds, n_codes)
    # property: dV is the exact integer products of the kernel's own codes, dequantised
    dV_codes = np.zeros_like(g["dV"], dtype=np.float64)
    for b in range(w.B):
        for h in range(w.H):
            for (i, j) in visited_blocks(N, causal):
                rows, cols = slice(64 * i, 64 * i + 64), slice(64 * j, 64 * j + 64)
                pc = dmp["P"][b, h, rows, cols].astype(np.int64)
                prod = pc.T @ dmp["dOh"][b, h, rows].astype(np.int64)
                dV_codes[b, h, cols] += float(dmp["sP"][b, h, i, j]) * float(dmp["sdO"][b, h, i]) * prod
    assert rel_l2(g["dV"], dV_codes) <= 1e-5
