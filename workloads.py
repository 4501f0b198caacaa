"""Seeded synthetic workloads for SageBwd attention (inputs only, no attention arithmetic).

This module is shared by the tests, the benchmark and the CPU oracle's callers.  It draws
Q, K, V and dO with numpy's ``default_rng(seed)`` as float32, in the order Q, K, V, dO, then
applies the per-workload structure (QK-norm, channel offsets, outlier channels) and rounds
every value to the workload's 16-bit dtype with round-to-nearest-even.  Arrays come back as
float32 holding exactly representable fp16/bf16 values, shape (B, H, N, d).

Workloads (sizes and distributions follow the SageBwd pages' synthetic set-ups; where a
"N(0, v)" is given, v is the variance):

  tiny      B1 H1  N128   d64  fp16, non-causal; Q,K,V,dO ~ N(0,1)
  sweep     B1 H8  N1024  d128 fp16, non-causal; Q,K ~ N(0, sigma^2), V,dO ~ N(0,1)
            (the random-QKV sigma sweep of "SageBwd: A Trainable Low-bit Attention", Table 1)
  qknorm    B4 H16 N4096  d128 bf16, causal; Q,K RMS-normalised per token (gamma=1,
            eps=1e-6), then K + per-(head, channel) offset ~ N(0,4); V ~ N(0,1); dO ~ N(0,1e-4)
  outlier   B2 H32 N8192  d64  fp16, causal; Q,K,V ~ N(0,1) with one channel per head
            (ceil(1% of d)) scaled x10 in each of Q, K, V; dO ~ N(0,1e-4)
  longseq   B1 H8  N32768 d128 bf16, causal; QK-normed Q,K; V ~ N(0,1); dO ~ N(0,1e-5)
  headline  B2 H16 N8192  d128 fp16; Q,K,V ~ N(0,1); dO ~ N(0,1e-4) (non-causal and causal)

QK-norm ("SageBwd: A Trainable Low-bit Attention", prerequisites, QK-norm paragraph) is
x / sqrt(mean(x^2) + eps) * gamma with gamma = 1 and the pages' norm epsilon 1e-6.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "fp16" | "bf16"
    causal: bool
    qk: str = "normal"    # "normal" | "qknorm" | "outlier"
    sigma: float = 1.0    # std of Q and K draws (before any QK-norm)
    k_offset_var: float = 0.0
    do_var: float = 1.0
    smooth_q: bool = False

    @property
    def tag(self) -> str:
        return f"B{self.B} H{self.H} N{self.N} d{self.d} {self.dtype} {'causal' if self.causal else 'non-causal'}"


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, "fp16", False),
    "sweep": Workload("sweep", 1, 8, 1024, 128, "fp16", False),
    "qknorm": Workload("qknorm", 4, 16, 4096, 128, "bf16", True, qk="qknorm",
                       k_offset_var=4.0, do_var=1e-4),
    "outlier": Workload("outlier", 2, 32, 8192, 64, "fp16", True, qk="outlier", do_var=1e-4),
    "longseq": Workload("longseq", 1, 8, 32768, 128, "bf16", True, qk="qknorm", do_var=1e-5),
    "headline": Workload("headline", 2, 16, 8192, 128, "fp16", False, do_var=1e-4),
}

SWEEP_SIGMAS = (1.0, 3.0, 5.0, 8.0, 10.0)


def get(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def round_fp16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest fp16 (ties to even) and return them as float32."""
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even) and return them as float32."""
    x = np.ascontiguousarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp16":
        return round_fp16(x)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(dtype)


def _qknorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    ms = np.mean(x.astype(np.float64) ** 2, axis=-1, keepdims=True)
    return (x / np.sqrt(ms + eps)).astype(np.float32)


def make_inputs(w: Workload, seed: int = 0, heads: int | None = None):
    """Return dict(Q, K, V, dO) of float32 arrays (B, H, N, d) holding dtype-exact values.

    ``heads`` limits H (the draws are then those of a workload with that many heads; used for
    small CPU-side samples of a large workload).
    """
    H = w.H if heads is None else heads
    shape = (w.B, H, w.N, w.d)
    rng = np.random.default_rng(seed)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    do = rng.standard_normal(shape, dtype=np.float32)
    if w.sigma != 1.0:
        q *= np.float32(w.sigma)
        k *= np.float32(w.sigma)
    if w.qk == "qknorm":
        q = _qknorm(q)
        k = _qknorm(k)
        if w.k_offset_var > 0:
            off = rng.standard_normal((1, H, 1, w.d), dtype=np.float32) * np.float32(math.sqrt(w.k_offset_var))
            k = k + off
    elif w.qk == "outlier":
        nch = max(1, math.ceil(0.01 * w.d))
        for t in (q, k, v):
            for h in range(H):
                ch = rng.choice(w.d, size=nch, replace=False)
                t[:, h, :, ch] *= np.float32(10.0)
    if w.do_var != 1.0:
        do *= np.float32(math.sqrt(w.do_var))
    return {name: round_to(t, w.dtype) for name, t in (("Q", q), ("K", k), ("V", v), ("dO", do))}
