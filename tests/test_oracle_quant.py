"""Pins for the oracle's quantiser and smoothing (CPU only).

The quantiser follows "SageBwd: A Trainable Low-bit Attention" (structured summary),
prerequisites, INT8 quantisation, and "SageAttention3 ..." (review) eq. (7); K-smoothing the
structured summary's K-/Q-smoothing paragraph.  Expected values come from hand-worked examples
(tests/golden) and from an exact rational re-derivation (tests/exact.py), never from the oracle.
"""
import os
from fractions import Fraction as Fr

import numpy as np
import pytest

from oracle import quant
from tests.exact import quantize_block_exact, fl32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantizer_worked_examples.txt")


def _golden_examples():
    lines = [l.strip() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    for k in range(0, len(lines), 3):
        blk = [float(v) for v in lines[k].split(":", 1)[1].split()]
        num, den = (int(v) for v in lines[k + 1].split(":", 1)[1].split())
        codes = [int(v) for v in lines[k + 2].split(":", 1)[1].split()]
        yield blk, Fr(num, den), codes


@pytest.mark.parametrize("blk,delta,codes", list(_golden_examples()))
def test_worked_examples(blk, delta, codes):
    q, d = quant.quantize_block(np.array(blk, np.float32))
    assert Fr(float(d)) == delta
    assert q.tolist() == codes
    # the exact re-derivation agrees with the hand-worked values too
    qe, de = quantize_block_exact(blk)
    assert qe == codes and de == delta


def _all_finite_fp16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16)
    return vals[np.isfinite(vals)].astype(np.float32)


def test_brute_force_every_fp16_value():
    """Every finite fp16 value, placed in blocks of 64 (in order and shuffled), quantises exactly
    as the rational re-derivation says."""
    vals = _all_finite_fp16()
    rng = np.random.default_rng(7)
    for arrangement in (vals, rng.permutation(vals)):
        n = (arrangement.size // 64) * 64
        blocks = arrangement[:n].reshape(-1, 64)
        # scale some blocks down so that small maxima and subnormal scales are exercised
        for k, blk in enumerate(blocks):
            if k % 3 == 1:
                blk = (blk * np.float32(2.0 ** -20)).astype(np.float32)
            q, d = quant.quantize_block(blk)
            qe, de = quantize_block_exact([Fr(float(v)) for v in blk])
            assert Fr(float(d)) == de, k
            assert q.tolist() == qe, k


def test_zero_block_and_tiny_block():
    q, d = quant.quantize_block(np.zeros(64, np.float32))
    assert d == 0 and not q.any()
    # max|x| / 127 underflows to zero in float32: zero-block rule
    tiny = np.zeros(64, np.float32)
    tiny[3] = np.float32(2.0 ** -149)
    q, d = quant.quantize_block(tiny)
    assert d == 0 and not q.any()


def test_codes_symmetric_range():
    x = np.linspace(-5, 5, 64).astype(np.float32)
    q, d = quant.quantize_block(x)
    assert q.min() == -127 and q.max() == 127
    assert np.all(np.abs(x - d * q.astype(np.float32)) <= d / 2 * (1 + 1e-6))


def test_per_block_layout():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 3, 256, 16)).astype(np.float32)
    x[1, 2, 64:128] *= 100
    q, s = quant.quantize_per_block(x)
    assert q.shape == x.shape and s.shape == (2, 3, 4)
    for b in range(2):
        for h in range(3):
            for i in range(4):
                qe, de = quantize_block_exact([Fr(float(v)) for v in x[b, h, 64 * i:64 * i + 64].ravel()])
                assert Fr(float(s[b, h, i])) == de
                assert q[b, h, 64 * i:64 * i + 64].ravel().tolist() == qe


def test_k_mean_is_exact_mean_rounded_once():
    rng = np.random.default_rng(2)
    k = rng.standard_normal((1, 2, 128, 8)).astype(np.float16).astype(np.float32) * np.float32(3)
    mu = quant.k_mean(k)
    for h in range(2):
        for c in range(8):
            exact = sum(Fr(float(v)) for v in k[0, h, :, c]) / 128
            assert Fr(float(mu[0, h, c])) == fl32(exact)


def test_q_block_mean_is_exact_mean_rounded_once():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 128, 4)).astype(np.float16).astype(np.float32)
    mu = quant.q_block_mean(q)
    assert mu.shape == (1, 1, 2, 4)
    for i in range(2):
        for c in range(4):
            exact = sum(Fr(float(v)) for v in q[0, 0, 64 * i:64 * i + 64, c]) / 64
            assert Fr(float(mu[0, 0, i, c])) == fl32(exact)


def test_quantize_smooth_reconstructs_inputs():
    """K^ delta_K + mu_K stays within half a quantisation step (plus float32 rounding) of K."""
    rng = np.random.default_rng(4)
    shape = (1, 2, 128, 32)
    Q, K, V = (rng.standard_normal(shape).astype(np.float16).astype(np.float32) for _ in range(3))
    K += np.float32(5)            # a large shared offset that K-smoothing removes
    out = quant.quantize_smooth(Q, K, V, smooth_k=True, smooth_q=True)
    muK = out["muK"]
    assert np.allclose(muK, K.mean(axis=2), atol=1e-5)
    for name, X, mean in (("K", K, muK[:, :, None, :]), ("V", V, 0.0)):
        codes, scales = out[name + "h"], out["s" + name]
        step = np.repeat(scales, 64, axis=2)[..., None]
        rec = codes.astype(np.float64) * step + mean
        assert np.all(np.abs(rec - X) <= step / 2 + 1e-5 * np.abs(X) + 1e-6)
    # smoothing shrinks K's scales: the offset is gone
    _, sK_raw = quant.quantize_per_block(K)
    assert np.all(out["sK"] < sK_raw / 2)
    # Q-smoothing: each block of Q_sm has (float32-rounded) zero mean
    qsm = out["Qh"].astype(np.float64) * np.repeat(out["sQ"], 64, axis=2)[..., None]
    assert np.abs(qsm.reshape(1, 2, 2, 64, 32).mean(axis=3)).max() < np.max(out["sQ"])
