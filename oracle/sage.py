"""Oracle: SageBwd forward and backward (TEST INFRASTRUCTURE, not product code).

The algorithm is taken in the pages' order and notation:

Forward -- "SageBwd: A Trainable Low-bit Attention" (structured summary), method steps,
forward (1)-(5); "SageAttention3 ..." (review), eq. (1) (online softmax) and eq. (8)
(INT8 forward: S_ij = MM(Q^_i, K^_j) s_Q s_K, per-token P with s_P = exp(rowmax(S_ij) - m_ij)/127,
O_ij update); section summary A.1 (returns O and the log-sum-exp L).

Backward -- "SageBwd: A Trainable Low-bit Attention" (structured summary), method steps,
backward (1)-(7); "SageAttention3 ..." (review), INT8 backward (Algorithm 3 equations): dV, dP kept
16-bit, dS = P o (dP - D), dQ, dK with per-block INT8 products; section summary A.2.

Readings where the pages are silent, garbled or at odds:
  R1  the softmax scale 1/sqrt(d) is applied after dequantisation, in float32, folded with
      log2(e) into c = fl32(fl32(s_Q s_K) * fl32(log2(e)/sqrt(d))).  The logits are float32
      values in log2 units, S_k = fl32(acc_k * c) (with Q-smoothing S_k = fl32(fl32(acc_k * c) +
      bias_k)); dQ and dK carry 1/sqrt(d) by the chain rule.
  R7  forward P^ is per token per 64-key tile: with r = max_k S_k the row max over the tile's
      unmasked entries and x_k = fl32(S_k - r), P^_k = rne(fl32(127 * fl32(2^x_k))), where 2^x
      is the float32 nearest to the exact power; s_P = 2^(r - m)/127; l accumulates the
      unquantised P~ (eq. 1); eq. (8)'s inverted rescale "diag(...)^-1" is read as eq. (1)'s
      non-inverted one.
  R8  backward P_k = fl32(2^(fl32(S_k - L2))) with L2 = fl32(L * fl32(log2(e))); P and dS are
      quantised per 64x64 tile: s = fl32(max|x|/127), its reciprocal inv = fl32(1/s) formed once
      per tile, q = clamp(rne(fl32(x * inv)), -127, 127) (the pages say only "round"); a tile
      whose max|x| is below 2^-120 (zero, or so small that 1/s is not a finite float32) gets
      s = 0, q = 0.
  R9  dP = dO V^T uses the unquantised 16-bit dO and V, float32 result, never rounded to 16 bits.
  R10 D = rowsum(dO o O) uses the stored 16-bit O.
  R11 no K-smoothing correction in the backward pass.
  R12 causal = top-left-aligned mask (key index <= query index); fully masked tiles are skipped.
  R13 L is natural-log, float32, in units of the scaled logits.
  R5  with Q-smoothing, S gets the bias mu_Qi K_sm,j^T (before 1/sqrt(d)) and dK gets
      (dS_ij^T 1) mu_Qi^T / sqrt(d) from the unquantised dS.

Where float decides an integer code (P^, dS^), the decision is taken in float32, each named
step one correctly rounded float32 operation; everything that only accumulates (m, l, O, dV,
dQ, dK, D) is float64.

FP8 variant (``QUANTISED_FP8``; "SageAttention3 ..." (review), "INT8 vs FP8 training"): every
INT8 code becomes an E4M3 code with 448 in place of 127 (see oracle.quant): block scales
fl32(max|x|/448); forward P^_k = e4m3_round(fl32(448 * fl32(2^x_k))), s_P = 2^(r - m)/448;
backward tile codes e4m3_round(fl32(x * fl32(1/s))), s = fl32(max|x|/448), a tile whose max|x|
is below 2^-110 being a zero tile (1/s stays finite).  Block products of E4M3 values are exact in
float64: each product is a multiple of 2^-18 below 2^18, a sum of at most 128 of them stays
below 2^25, so 43 bits suffice.  (Their logits fl32(acc * c) take one float64 rounding before the
float32 one, since acc * c may need 67 bits; integer products need at most 45 and are exact.)

The ``DEQUANTISED`` arithmetic replaces every quantiser by the identity and drops every float32
rounding; the very same tiled code must then equal float64 full-precision attention, which pins
the tiling, the online-softmax bookkeeping, L and the backward structure (tests/test_oracle_sage.py).
"""
from __future__ import annotations

import math

import numpy as np

from .quant import BLOCK, QMAX, e4m3_round, quantize_per_block, quantize_smooth, k_mean, q_block_mean

LOG2E = 1.4426950408889634      # log2(e), the double nearest 1/ln(2)
LN2 = 0.6931471805599453
F32 = np.float32
# R8b: a backward P / dS tile whose max|x| is below 2^-120 is a zero tile (s = 0, q = 0); below
# that bound the float32 reciprocal 1/s of its scale would overflow.
TILE_ZERO_BELOW = np.float32(2.0 ** -120)
TILE_ZERO_BELOW_FP8 = np.float32(2.0 ** -110)     # the same bound for s = max|x| / 448


class Arith:
    """The arithmetic of the quantisation steps: SageBwd's (quantised) or the identity limit."""

    def __init__(self, quantised: bool, fmt: str = "int8"):
        self.quantised = quantised
        self.fmt = fmt                  # code format: "int8" or "e4m3"
        self.qmax = QMAX[fmt]           # 127 or 448

    # -- plain float helpers --------------------------------------------------------------
    def r32(self, x):
        return np.asarray(x, np.float64).astype(np.float32) if self.quantised else np.asarray(x, np.float64)

    def scale_log2(self, d: int):
        return F32(LOG2E / math.sqrt(d)) if self.quantised else LOG2E / math.sqrt(d)

    def logit_scale(self, sq, sk, sl2):
        """c = fl32(fl32(s_Q s_K) * sl2): the float32 factor taking an integer product to log2 units."""
        if self.quantised:
            return F32(F32(sq) * F32(sk)) * F32(sl2)
        return float(sq) * float(sk) * float(sl2)

    # -- exact integer block products ------------------------------------------------------
    def int_mm(self, a, b):
        """MM(A^, B^): exact for integer codes (every partial sum is far below 2^53) and for E4M3
        codes (multiples of 2^-18 below 2^25: checked)."""
        p = np.asarray(a, np.float64) @ np.asarray(b, np.float64)
        if not self.quantised:
            return p
        if self.fmt == "e4m3":
            assert np.array_equal(np.rint(p * 2.0 ** 18), p * 2.0 ** 18), "E4M3 block product not exact"
            return p
        r = np.rint(p)
        assert np.array_equal(r, p), "integer block product is not integral"
        return r.astype(np.int64)

    def logits(self, s_int, c, bias=None):
        """The logits in log2 units as float32 values (R1): S = fl32(acc * c), then with a bias
        S = fl32(S + bias).  acc * c of an integer product (|acc| < 2^21 times a 24-bit c) is
        exact in float64, so one cast rounds once."""
        acc = np.asarray(s_int, np.float64)
        if not self.quantised:
            return acc * c + (0.0 if bias is None else np.asarray(bias, np.float64)[None, :])
        S = (acc * float(F32(c))).astype(np.float32)
        if bias is not None:
            S = S + np.asarray(bias, np.float32)[None, :]        # float32 add, one rounding
        return S

    def minus(self, S, sub):
        """x = fl32(S - sub) with ``sub`` one value per row (a row max r or L2)."""
        if not self.quantised:
            return np.asarray(S, np.float64) - np.asarray(sub, np.float64)[:, None]
        return (np.asarray(S, np.float32) - np.asarray(sub, np.float32)[:, None]).astype(np.float32)

    @staticmethod
    def row_max(S, valid):
        """r = the row max of S over ``valid`` entries, -inf where a row has none."""
        return np.where(valid, S, -np.inf).max(axis=1)

    # -- the quantisers --------------------------------------------------------------------
    def block_quant(self, x):
        """Per-64-token-block quantiser of Q, K, V, dO (see oracle.quant)."""
        if self.quantised:
            return quantize_per_block(x, fmt=self.fmt)
        x = np.asarray(x, np.float64)
        return x, np.ones(x.shape[:-2] + (x.shape[-2] // BLOCK,))

    def token_quant(self, x, unrounded: bool = False):
        """Forward per-token P^ of one tile (R7) from x = logits - r.
        Returns (2^x in float64, P^), and with ``unrounded`` also the float32 values
        fl32(127 * fl32(2^x)) that the rounding decides from."""
        e64 = np.exp2(np.asarray(x, np.float64))
        if not self.quantised:
            y = 127.0 * e64
            return (e64, y, y) if unrounded else (e64, y)
        e32 = e64.astype(np.float32)
        y = (F32(self.qmax) * e32).astype(np.float32)
        if self.fmt == "e4m3":
            q = e4m3_round(y)
        else:
            q = np.clip(np.rint(y), 0, 127).astype(np.int64)
        return (e64, q, y) if unrounded else (e64, q)

    def tile_quant(self, x, unrounded: bool = False):
        """Backward per-tile quantiser of P and dS (R8).  Returns (scale, codes), and with
        ``unrounded`` also the float32 values fl32(x * inv) that the rounding decides from."""
        if not self.quantised:
            x = np.asarray(x, np.float64)
            return (1.0, x, x) if unrounded else (1.0, x)
        x = np.asarray(x, np.float32)
        mx = np.max(np.abs(x)) if x.size else F32(0)
        zero = mx < (TILE_ZERO_BELOW_FP8 if self.fmt == "e4m3" else TILE_ZERO_BELOW)
        if zero:
            s, inv = F32(0), F32(0)
        else:
            s = F32(mx) / F32(self.qmax)
            inv = F32(1) / s
        y = (x * inv).astype(np.float32)                     # float32 product, one rounding
        if self.fmt == "e4m3":
            q = e4m3_round(y)
        else:
            q = np.clip(np.rint(y), -127, 127).astype(np.int64)   # rint: ties to even
        return (s, q, y) if unrounded else (s, q)

    def exp2_32(self, x):
        if self.quantised:
            return np.exp2(np.asarray(x, np.float32).astype(np.float64)).astype(np.float32)
        return np.exp2(np.asarray(x, np.float64))


QUANTISED = Arith(True)
QUANTISED_FP8 = Arith(True, fmt="e4m3")
DEQUANTISED = Arith(False)


def prepare(Q, K, V, smooth_k: bool = True, smooth_q: bool = False, arith: Arith = QUANTISED) -> dict:
    """Steps a1 + a2 in the chosen arithmetic: K-mean, smoothing and the per-block quantisers."""
    if arith.quantised:
        return quantize_smooth(Q, K, V, smooth_k=smooth_k, smooth_q=smooth_q, fmt=arith.fmt)
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    B, H, N, d = K.shape
    ones = np.ones((B, H, N // BLOCK))
    muK = K.mean(axis=-2) if smooth_k else np.zeros((B, H, d))
    Ksm = K - muK[:, :, None, :]
    if smooth_q:
        muQ = Q.reshape(B, H, N // BLOCK, BLOCK, d).mean(axis=-2)
        Qsm = (Q.reshape(B, H, N // BLOCK, BLOCK, d) - muQ[:, :, :, None, :]).reshape(B, H, N, d)
    else:
        muQ, Qsm = None, Q
    return dict(Qh=Qsm, Kh=Ksm, Vh=V, sQ=ones, sK=ones.copy(), sV=ones.copy(), muK=muK, muQ=muQ, Ksm=Ksm)


def _bias_log2(prep, b, h, i, sl2, arith: Arith):
    """Q-smoothing bias of query block i in log2 units: fl32(fl32(mu_Qi . K_sm[n]) * sl2) per key n."""
    mu = np.asarray(prep["muQ"][b, h, i], np.float64)
    ksm = np.asarray(prep["Ksm"][b, h], np.float64)
    bias = ksm @ mu
    if arith.quantised:
        return bias.astype(np.float32) * F32(sl2)
    return bias * sl2


def _causal_mask(n: int) -> np.ndarray:
    """True where a key lies after the query inside a diagonal tile (top-left aligned)."""
    return np.triu(np.ones((n, n), bool), k=1)


def sage_forward(prep: dict, causal: bool, arith: Arith = QUANTISED, q_blocks=None, heads=None,
                 record: dict | None = None):
    """SageBwd forward (steps a3-a6).  Returns (O float64 (B,H,N,d), L float64 (B,H,N)).

    ``q_blocks`` limits the query blocks computed (others stay zero), ``heads`` the (b, h) pairs.
    ``record`` (small N only) receives, per head, the S block products, the float32 logits S and
    the products acc c they are rounded from, the P^ codes, the float32 values their rounding decides from (P_y) and the P^ V^ block products of
    every tile (integers for INT8 codes, float64 for E4M3).
    """
    Qh, Kh, Vh = prep["Qh"], prep["Kh"], prep["Vh"]
    sQ, sK, sV = prep["sQ"], prep["sK"], prep["sV"]
    B, H, N, d = Qh.shape
    T = N // BLOCK
    sl2 = arith.scale_log2(d)
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    mask = _causal_mask(BLOCK)
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for (b, h) in heads:
        if record is not None:
            rec = record.setdefault((b, h), {})
            rtype = np.int64 if arith.fmt == "int8" else np.float64
            rec["S_int"] = np.zeros((N, N), rtype)
            rec["S"] = np.zeros((N, N), np.float32)
            rec["acc_c"] = np.zeros((N, N))
            rec["P_hat"] = np.zeros((N, N), rtype)
            rec["P_y"] = np.zeros((N, N), np.float32)
            rec["PV_int"] = {}
        for i in (range(T) if q_blocks is None else q_blocks):
            rows = slice(i * BLOCK, (i + 1) * BLOCK)
            m = np.full(BLOCK, -np.inf)
            l = np.zeros(BLOCK)
            acc = np.zeros((BLOCK, d))
            bias = _bias_log2(prep, b, h, i, sl2, arith) if prep.get("muQ") is not None else None
            for j in range(T):
                if causal and j > i:
                    break
                cols = slice(j * BLOCK, (j + 1) * BLOCK)
                # (3) S_ij = MM(Q^_i, K^_j) * s_Q * s_K  (and * 1/sqrt(d), in log2 units)
                s_int = arith.int_mm(Qh[b, h, rows], np.swapaxes(Kh[b, h, cols], 0, 1))
                c = arith.logit_scale(sQ[b, h, i], sK[b, h, j], sl2)
                S = arith.logits(s_int, c, None if bias is None else bias[cols])
                valid = ~mask if (causal and j == i) else np.ones((BLOCK, BLOCK), bool)
                # (4) online softmax statistics and per-token quantisation of P~
                r = arith.row_max(S, valid)
                x = arith.minus(S, np.where(np.isfinite(r), r, 0))
                x = np.where(valid, x, -np.inf)
                m_new = np.maximum(m, np.asarray(r, np.float64))
                e64, p_hat, p_y = arith.token_quant(x, unrounded=True)
                alpha = np.exp2(m - m_new)
                grow = np.exp2(np.asarray(r, np.float64) - m_new)
                s_p = grow / arith.qmax
                l = alpha * l + grow * e64.sum(axis=1)
                # (5) O_ij = diag(e^{m_old - m_new}) O + MM(P^_ij, V^_j) * s_P * s_V
                pv = arith.int_mm(p_hat, Vh[b, h, cols])
                acc = alpha[:, None] * acc + (s_p * float(sV[b, h, j]))[:, None] * pv
                m = m_new
                if record is not None:
                    rec["S_int"][rows, cols] = s_int
                    rec["S"][rows, cols] = S
                    rec["acc_c"][rows, cols] = np.asarray(s_int, np.float64) * float(c)
                    rec["P_hat"][rows, cols] = p_hat
                    rec["P_y"][rows, cols] = p_y
                    rec["PV_int"][(i, j)] = pv
            O[b, h, rows] = acc / l[:, None]
            L[b, h, rows] = (m + np.log2(l)) * LN2
    return O, L


def sage_backward(prep: dict, O_stored, L, dO, causal: bool, arith: Arith = QUANTISED,
                  q_blocks=None, kv_blocks=None, heads=None, record: dict | None = None,
                  dp_int8: bool = False, products: bool = False):
    """SageBwd backward (steps a7-a13).  Returns dict(dQ, dK, dV float64 (B,H,N,d), D, dOh, sdO).

    ``dp_int8`` selects the ablation of "SageAttention3 ..." (review), Table 1c: dP from the INT8
    codes of dO and V, dP_ij = fl32(MM(dO^_i, V^_j^T) * fl32(s_dO,i * s_V,j)), instead of the 16-bit
    product the method keeps.

    ``O_stored`` is the forward output as stored (16-bit values), ``L`` the stored float32 LSE.
    ``q_blocks`` / ``kv_blocks`` restrict which dQ rows / dK, dV rows are completed (for sampled
    checks at large N); by default everything is computed, looping over key/value blocks and,
    inside, query blocks.  ``record`` receives, per head, the per-tile dequantised P, dP and
    dequantised dS, the P and dS codes, the float32 values their rounding decides from (P_y, dS_y),
    the logits (S_bwd) and acc c (acc_c_bwd), and the tile scales (sP, sdS); with ``products`` also the integer block
    products MM(P^^T, dO^_i), MM(dS^, K^_j) and MM(dS^^T, Q^_i) of every tile (i, j).
    """
    if dp_int8 and arith.fmt != "int8":
        raise ValueError("the INT8-dP ablation applies to INT8 codes only")
    Qh, Kh = prep["Qh"], prep["Kh"]
    sQ, sK = prep["sQ"], prep["sK"]
    B, H, N, d = Qh.shape
    T = N // BLOCK
    sl2 = arith.scale_log2(d)
    inv_sqrt_d = 1.0 / math.sqrt(d)
    if "V16" not in prep:
        raise ValueError("prep must carry the unquantised 16-bit V as prep['V16']")
    V64 = np.asarray(prep["V16"], np.float64)
    dO = np.asarray(dO, np.float32)
    O64 = np.asarray(O_stored, np.float64)
    # (1) D = rowsum(dO o O) from the cached forward output
    D = (dO.astype(np.float64) * O64).sum(axis=-1)
    D32 = arith.r32(D)
    dOh, sdO = arith.block_quant(dO)
    L2 = arith.r32(np.asarray(L, np.float32 if arith.quantised else np.float64) * (F32(LOG2E) if arith.quantised else LOG2E))
    dQ = np.zeros((B, H, N, d))
    dK = np.zeros((B, H, N, d))
    dV = np.zeros((B, H, N, d))
    mask = _causal_mask(BLOCK)
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]

    def tile(b, h, i, j, bias, want_dq, want_dkv):
        rows = slice(i * BLOCK, (i + 1) * BLOCK)
        cols = slice(j * BLOCK, (j + 1) * BLOCK)
        # (2) recompute S_ij (same formula as the forward) and P_ij = exp(S_ij - L_i)
        s_int = arith.int_mm(Qh[b, h, rows], np.swapaxes(Kh[b, h, cols], 0, 1))
        c = arith.logit_scale(sQ[b, h, i], sK[b, h, j], sl2)
        S = arith.logits(s_int, c, None if bias is None else bias[cols])
        x = arith.minus(S, L2[b, h, rows])
        if causal and i == j:
            x = np.where(mask, -np.inf, x)
        P = arith.exp2_32(x)
        # (3) dV_j += MM(P^_ij^T, dO^_i) * s_P * s_dO
        s_p, p_hat, p_y = arith.tile_quant(P, unrounded=True)
        dv_int = arith.int_mm(p_hat.T, dOh[b, h, rows]) if (want_dkv or products) else None
        if want_dkv:
            dV[b, h, cols] += (float(s_p) * float(sdO[b, h, i])) * dv_int
        # (4) dP_ij = dO_i V_j^T, 16-bit operands, float32 result (ablation: INT8 codes, exact
        # integer product times the float32 product of the two block scales)
        if dp_int8:
            sc = arith.r32(np.float64(arith.r32(float(sdO[b, h, i]) * float(prep["sV"][b, h, j]))))
            dP = arith.r32(arith.int_mm(dOh[b, h, rows], np.swapaxes(prep["Vh"][b, h, cols], 0, 1)) * float(sc))
        else:
            dP = arith.r32(dO[b, h, rows].astype(np.float64) @ V64[b, h, cols].T)
        # (5) dS_ij = P_ij o (dP_ij - D_i), then per-tile quantisation
        dS = arith.r32(P * arith.r32(dP - D32[b, h, rows][:, None]))
        s_ds, ds_hat, ds_y = arith.tile_quant(dS, unrounded=True)
        # (6) dQ_i += MM(dS^_ij, K^_j) * s_dS * s_K   (and * 1/sqrt(d))
        dq_int = arith.int_mm(ds_hat, Kh[b, h, cols]) if (want_dq or products) else None
        if want_dq:
            dQ[b, h, rows] += (float(s_ds) * float(sK[b, h, j]) * inv_sqrt_d) * dq_int
        # (7) dK_j += MM(dS^_ij^T, Q^_i) * s_dS * s_Q   (and * 1/sqrt(d))
        dk_int = arith.int_mm(ds_hat.T, Qh[b, h, rows]) if (want_dkv or products) else None
        if want_dkv:
            dK[b, h, cols] += (float(s_ds) * float(sQ[b, h, i]) * inv_sqrt_d) * dk_int
            if prep.get("muQ") is not None:
                colsum = np.asarray(dS, np.float64).sum(axis=0)
                dK[b, h, cols] += inv_sqrt_d * np.outer(colsum, np.asarray(prep["muQ"][b, h, i], np.float64))
        if record is not None:
            rec = record.setdefault((b, h), {})
            for key in ("P", "dP", "dS"):
                rec.setdefault(key, np.zeros((N, N)))
            ctype = np.int64 if arith.fmt == "int8" else np.float64
            for key in ("P_hat", "dS_hat"):
                rec.setdefault(key, np.zeros((N, N), ctype))
            for key in ("P_y", "dS_y", "S_bwd"):
                rec.setdefault(key, np.zeros((N, N), np.float32))
            rec.setdefault("acc_c_bwd", np.zeros((N, N)))
            for key in ("sP", "sdS"):
                rec.setdefault(key, np.zeros((T, T), np.float32))
            rec["P"][rows, cols] = float(s_p) * np.asarray(p_hat, np.float64)
            rec["dP"][rows, cols] = dP
            rec["dS"][rows, cols] = float(s_ds) * np.asarray(ds_hat, np.float64)
            rec["P_hat"][rows, cols] = p_hat
            rec["dS_hat"][rows, cols] = ds_hat
            rec["P_y"][rows, cols] = p_y
            rec["dS_y"][rows, cols] = ds_y
            rec["S_bwd"][rows, cols] = S
            rec["acc_c_bwd"][rows, cols] = np.asarray(s_int, np.float64) * float(c)
            rec["sP"][i, j] = s_p
            rec["sdS"][i, j] = s_ds
            if products:
                rec.setdefault("dV_int", {})[(i, j)] = dv_int
                rec.setdefault("dQ_int", {})[(i, j)] = dq_int
                rec.setdefault("dK_int", {})[(i, j)] = dk_int

    for (b, h) in heads:
        biases = {}
        def bias_of(i):
            if prep.get("muQ") is None:
                return None
            if i not in biases:
                biases[i] = _bias_log2(prep, b, h, i, sl2, arith)
            return biases[i]
        if q_blocks is None and kv_blocks is None:
            for j in range(T):
                for i in range(j if causal else 0, T):
                    tile(b, h, i, j, bias_of(i), True, True)
        else:
            for j in (kv_blocks or []):
                for i in range(j if causal else 0, T):
                    tile(b, h, i, j, bias_of(i), False, True)
            for i in (q_blocks or []):
                for j in range(0, (i + 1) if causal else T):
                    tile(b, h, i, j, bias_of(i), True, False)
    return dict(dQ=dQ, dK=dK, dV=dV, D=D, dOh=dOh, sdO=sdO)


def run(Q, K, V, dO, causal: bool, dtype_round, smooth_k: bool = True, smooth_q: bool = False,
        arith: Arith = QUANTISED, record: dict | None = None, dp_int8: bool = False,
        products: bool = False):
    """Whole path on full tensors: quantise, forward, backward.  ``dtype_round`` rounds O to the
    stored 16-bit type (identity in the dequantised limit)."""
    prep = prepare(Q, K, V, smooth_k=smooth_k, smooth_q=smooth_q, arith=arith)
    prep["V16"] = np.asarray(V, np.float64)
    O, L = sage_forward(prep, causal, arith=arith, record=record)
    O_stored = dtype_round(O.astype(np.float32)) if arith.quantised else O
    L_stored = L.astype(np.float32) if arith.quantised else L
    g = sage_backward(prep, O_stored, L_stored, dO, causal, arith=arith, record=record, dp_int8=dp_int8,
                      products=products)
    return dict(prep=prep, O=O, L=L, O_stored=O_stored, L_stored=L_stored, **g)
