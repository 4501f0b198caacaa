"""Pin of the quantised oracle's per-block scale bookkeeping (CPU only).

"SageBwd: A Trainable Low-bit Attention" (structured summary), prerequisites "INT8 quantisation"
and method steps, forward (3), (5) and backward (3), (6), (7); "SageAttention3 ..." (review),
eq. (7): every integer block product is dequantised with the scales of exactly the blocks it
multiplies -- S_ij with s_Q,i s_K,j, O with s_P s_V,j, dV_j with s_P,ij s_dO,i, dQ_i with
s_dS,ij s_K,j, dK_j with s_dS,ij s_Q,i.

The dequantised limit (every scale 1) cannot see an index mistake in that bookkeeping, so here
every 64-token block of Q, K, V and dO is integer codes (one of them 127) times its own power of
two: the block quantiser then returns those codes and that power exactly, the blocks' scales differ
by up to 2^12, and the only quantisation left is the per-token P of the forward and the per-tile P
and dS of the backward.  The quantised oracle (no smoothing, so that K^ is exact) must then stay
within rel-l2 0.1 of float64 full-precision attention (oracle.fpa, itself pinned by finite
differences); it measures at most 0.043.  The mutation test plants each plausible mistake in a copy
of the oracle's source (a scale taken from the wrong block) and checks that the pin fails: the
mutated gradients measure 0.31 or more.
"""
import types

import numpy as np
import pytest

import workloads
from oracle import fpa, metrics, sage

GATE = 0.1
SHAPE = (1, 2, 256, 64)


def _block_codes(rng, shape, exps):
    """Integer codes in [-127, 127] (normal, std 40, one 127 per 64-token block), each block times
    2^exps[block]: values that are exact in fp16 and that the block quantiser reproduces."""
    codes = np.clip(np.rint(rng.standard_normal(shape) * 40), -127, 127)
    codes[..., ::64, 0] = 127.0
    per_token = np.repeat(2.0 ** np.asarray(exps, np.float64), 64)
    return (codes * per_token[None, None, :, None]).astype(np.float32)


def _case(trial):
    """Q, K block exponents in [-8, -5] (logits of a few units), V and dO in [-6, 6]."""
    rng = np.random.default_rng(7 + trial)
    T = SHAPE[2] // 64
    eq, ek = rng.integers(-8, -4, T), rng.integers(-8, -4, T)
    ev, edo = rng.integers(-6, 7, T), rng.integers(-6, 7, T)
    return tuple(_block_codes(rng, SHAPE, e) for e in (eq, ek, ev, edo))


CASES = [(trial, causal) for trial in range(2) for causal in (False, True)]


def _errors(mod, Q, K, V, dO, causal):
    out = mod.run(Q, K, V, dO, causal, workloads.round_fp16, smooth_k=False)
    O, _, _ = fpa.fpa_forward(Q, K, V, causal)
    g = fpa.fpa_backward(Q, K, V, dO, causal)
    errs = {k: metrics.rel_l2(out[k], g[k]) for k in ("dQ", "dK", "dV")}
    errs["O"] = metrics.rel_l2(out["O"], O)
    return errs


def test_block_codes_are_exact():
    Q, K, V, dO = _case(0)
    for x in (Q, K, V, dO):
        assert np.array_equal(workloads.round_fp16(x), x)
        codes, scales = sage.QUANTISED.block_quant(x)
        back = codes.astype(np.float64) * np.repeat(scales, 64, axis=-1)[..., None]
        assert np.array_equal(back, x.astype(np.float64))
        assert len(np.unique(scales)) > 1


@pytest.mark.parametrize("trial,causal", CASES)
def test_block_scaled_inputs_match_fpa(trial, causal):
    errs = _errors(sage, *_case(trial), causal)
    for k, e in errs.items():
        assert e < GATE, (k, e)


# (name, the oracle's line, the mistake planted in it)
MUTATIONS = [
    ("dK with s_K,j in place of s_Q,i", "dK",
     "(float(s_ds) * float(sQ[b, h, i]) * inv_sqrt_d) * dk_int",
     "(float(s_ds) * float(sK[b, h, j]) * inv_sqrt_d) * dk_int"),
    ("dV with s_dO of key block j", "dV",
     "(float(s_p) * float(sdO[b, h, i])) * dv_int",
     "(float(s_p) * float(sdO[b, h, j])) * dv_int"),
    ("dQ with s_Q,i in place of s_K,j", "dQ",
     "(float(s_ds) * float(sK[b, h, j]) * inv_sqrt_d) * dq_int",
     "(float(s_ds) * float(sQ[b, h, i]) * inv_sqrt_d) * dq_int"),
    ("O with s_V of query block i", "O",
     "(s_p * float(sV[b, h, j]))[:, None] * pv",
     "(s_p * float(sV[b, h, i]))[:, None] * pv"),
    ("S with the scales' blocks swapped", "O",
     "c = arith.logit_scale(sQ[b, h, i], sK[b, h, j], sl2)\n                S = arith.logits(",
     "c = arith.logit_scale(sQ[b, h, j], sK[b, h, i], sl2)\n                S = arith.logits("),
]


def _mutated_oracle(old: str, new: str):
    """A copy of oracle/sage.py with ``old`` replaced by ``new``, loaded as a module of the oracle
    package (so that its relative imports resolve)."""
    src = open(sage.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle._mutated_sage")
    mod.__package__ = "oracle"
    mod.__file__ = sage.__file__
    exec(compile(src.replace(old, new), sage.__file__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,target,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_scale_mistakes_fail_the_pin(name, target, old, new):
    mod = _mutated_oracle(old, new)
    worst = max(_errors(mod, *_case(trial), causal)[target] for trial, causal in CASES)
    assert worst > 3 * GATE, (name, worst)
