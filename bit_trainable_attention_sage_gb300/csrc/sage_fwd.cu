// sage_fwd.cu -- SageBwd forward on sm_103a tensor cores (tcgen05, TMA, TMEM).
//
// Method: "SageBwd: A Trainable Low-bit Attention" (structured summary), method steps, forward
// (3)-(5); "SageAttention3 ..." (review) eq. (1) (online softmax) and eq. (8) (INT8 forward:
// S_ij = MM(Q^_i, K^_j) s_Q s_K, per-token P codes with s_P = exp(rowmax(S_ij) - m_ij) / 127,
// O_ij = diag(e^{m_{i,j-1} - m_ij}) O_{i,j-1} + MM(P^_ij, V^_j) s_P s_V); section summary A.1
// (the forward returns O and the log-sum-exp L).
//
// GB300 design.  sm_103a has no INT8 tcgen05 MMA, so the int8 codes run through kind::f16 MMAs as
// integer-valued fp16: every |code| <= 127 is exact in fp16, every product <= 127^2 and every
// partial sum over a 128-long contraction <= 2 064 512 < 2^24 is exact in the fp32 accumulator,
// so the block products are the exact integers the method defines.
//
// One CTA owns two 128-row query tiles (four 64-row quantisation blocks) of one head and walks
// the keys in steps of 128 (two 64-key blocks); both tiles share every K and V tile it loads:
//   warp 8      TMA producer: both Q tiles once, then K and V tiles, double-buffered (step j in
//               stage j & 1; step j + 1's tiles stream in while step j's MMAs read the other)
//   warp 9      allocates TMEM; one lane issues every MMA, for each tile t:
//                 S_t    = Q^_t K^T                 M=128 N=128 K=d  -> TMEM cols 256t + [0,128)
//                 PV_t,h = P^_t[:,64h:64h+64] V^_h  M=128 N=d   K=64 -> TMEM cols 256t + [128,256)
//               (d = 64: half h into its own 64 columns 256t + 128 + 64h, so that PV_t,1 need
//               not wait for the O update that reads PV_t,0)
//   warps 0-3   softmax of tile 0, warps 4-7 of tile 1: thread = query row = TMEM lane.  Per step:
//               logits, row max per 64-key block, P codes (written back to TMEM over the consumed
//               S columns, as the A operand of the PV MMA), running max and sum, then
//               O = alpha O + s_P s_V PV_h in registers.
// While one warpgroup turns S into codes the tensor core works on the other tile, so the two
// softmax warpgroups and the MMA pipe overlap.  TMEM: all 512 columns; one CTA per SM.

// Numerics (the method's steps, with 2^x by the hardware approximation: a code can therefore
// differ from the one exact powers give only where 127 * 2^x lies within rounding distance of a
// half-integer).  The logit is rounded before r is subtracted, as the method forms S and then
// exponentiates S - r: fusing the two roundings moved the row sums l by up to 1e-5 relative at
// logits near 500 (sigma = 10 inputs), enough to change the 16-bit O and, through
// D = rowsum(dO o O), the backward's gradients by more than 1e-3.
//   c   = fl32(fl32(sQ_i sK_j) * fl32(log2(e)/sqrt(d)))
//   S_k = fl32(acc_k * c);  r = max_k S_k = fl32(max_k(acc_k) * c)   (64-key block, log2 units)
//   x_k = fl32(S_k - r)
//   P^_k = rint(127 * ex2(x_k))                  (the exact product, round half to even)
//   with Q-smoothing: S_k = fl32(fl32(acc_k * c) + bias_k), r = max S_k
//   l <- 2^(m - m') l + 2^(r - m') sum_k ex2(x_k);  O <- 2^(m - m') O + (2^(r - m') / 127) s_V PV
//   O_out = O / l;  L = (m + log2 l) ln 2
// FP8 variant (SAGE_FLAG_FP8, "SageAttention3 ..." (review), INT8 vs FP8 training): the codes are
// E4M3 values, P^_k = e4m3(fl32(448 * ex2(x_k))) and the PV scale is (2^(r - m') / 448) s_V.
// E4M3 values are exact fp16 operands; their products are exact in the fp32 accumulator, the
// sums rounded as any fp32 accumulation.
// FP4 inference forward ("SageAttention3 ..." (review), eq. (4)-(6)): Q, K, V arrive as their
// dequantised NVFP4 values s * code (exact fp16, at most 6 significant bits), so c = fl32(log2(e) /
// sqrt(d)) alone; P~2 = fl32(2688 ex2(x)) is quantised per 16 keys, s_P2 = e4m3(fl32(max / 6)),
// code = e2m1(fl32(v fl32(1 / s_P2))), and the PV operand is s_P2 * code; the PV scale is
// s_P1 = 2^(r - m') / 2688 (eq. (6) with the tile row max r).
// Attn-QAT forward ("Attn-QAT: 4-Bit Attention With Quantization-Aware Training", technical
// summary, section 2.2): Q, K, V arrive fake-quantised in the input 16-bit type, and the MMAs run
// on that type; c = fl32(log2(e) / sqrt(d)).  Two passes of this kernel: the first (QAT) codes
// P^ = phi(e), phi one-level NVFP4 per 16 keys (s = e4m3(fl32(max / 6)), code =
// e2m1(fl32(e fl32(1 / s))), operand s * code), and writes O, L and the row maxima r of every
// (key block, row), from which the backward rebuilds P^; the second (QAT_HP) feeds the
// unquantised e rounded to the 16-bit type and writes the high-precision O' in float32.  Both
// scale their PV products by 2^(r - m') alone.  (A fused pass would need a second O accumulator:
// 2 d float32 registers a thread do not fit beside the rest at d = 128.)
#include "sage_device.cuh"
#include "sage_internal.h"

namespace sage {

__device__ unsigned int g_fwd_err;

namespace fwd {

// warps 0-3: softmax of tile 0, 4-7: tile 1, 8: TMA producer, 9: MMA issuer, 10-11: idle.
// Launched at 168 registers a thread (384 x 168 = 64512); the control warpgroup gives registers
// back (40) and the softmax warpgroups take them (232): 2 x 128 x 232 + 128 x 40 = 64512.
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kRegsSoftmax = 232;
constexpr uint32_t kRegsControl = 40;

template <int D>
struct Smem {
    alignas(1024) uint8_t q[2][D / 64][128 * 128];   // [tile][chunk][row][64 halves], 128B swizzle
    alignas(1024) uint8_t k[2][D / 64][128 * 128];   // two stages: step j's tile in stage j & 1
    alignas(1024) uint8_t v[2][D / 64][128 * 128];
    uint64_t q_full, k_full[2], k_free[2], v_full[2], v_free[2], mma_done;
    uint64_t s_full[2], p_full[2][2];                  // p_full[tile][64-key half]
    uint64_t pv_full[2][D == 64 ? 2 : 1], pv_free[2][D == 64 ? 2 : 1];   // [tile][PV buffer]
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) { return pack2<__nv_bfloat16>(lo, hi); }

// number of keys a CTA tile visits: causal tiles stop at their last row
__device__ __forceinline__ int tile_kv_end(int q0, int N, int causal) {
    if (q0 >= N) return 0;
    return causal ? min(N, q0 + 128) : N;
}

// Row maximum of a 64-key block held in registers (of the integer products, or with Q-smoothing
// of the biased logits acc c + bias, which then replace the products in `raw`), masked to the
// first `nvalid` keys when MASKED.
template <bool BIAS, bool MASKED>
__device__ __forceinline__ float fwd_row_max(uint32_t (&raw)[64], float c, const float *bias,
                                             int nvalid) {
    float rp[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int k = 0; k < 64; k += 4) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float acc = __uint_as_float(raw[k + e]);
            v[e] = BIAS ? __fadd_rn(__fmul_rn(acc, c), bias[k + e]) : acc;   // S = fl32(fl32(acc c) + b)
            if (BIAS) raw[k + e] = __float_as_uint(v[e]);
            if (MASKED) v[e] = (k + e < nvalid) ? v[e] : -INFINITY;
        }
        rp[0] = max3f(rp[0], v[0], v[1]);
        rp[1] = max3f(rp[1], v[2], v[3]);
    }
    return fmaxf(rp[0], rp[1]);
}

// Codes of a 64-key block: P^ = rint(fl32(127 ex2(x))), x = fl32(S - r) with the logit
// S = fl32(acc c) (with Q-smoothing S = fl32(fl32(acc c) + bias), left in `raw` by the row
// maximum), packed as fp16 pairs into the 32 TMEM columns at `code_col`;
// returns the row sum of ex2(x) (four partial sums).  rint is a fused multiply-add of 1.5 * 2^23
// (float32 spacing 1 there, so the exact product 127 ex2(x) is rounded to an integer once) and an
// exact subtraction: full-rate instructions, unlike the conversion unit's round-to-integer.  This
// differs from rint(fl32(127 ex2(x))) only within 127 ex2(x) 2^-24 of a half-integer.
// FP8: P^ = e4m3(fl32(448 ex2(x))) instead, converted to fp16 in two instructions per pair.
// FP4: each 16-key group is an NVFP4 block of v = fl32(2688 ex2(x)) (two passes over the group:
// its maximum, then the codes), written as the dequantised fp16 values.
constexpr int kFmtInt8 = 0, kFmtFp8 = 1, kFmtFp4 = 2, kFmtQat = 3, kFmtQatHp = 4;
// formats whose block scales live inside the dequantised operands: c = log2(e)/sqrt(d) alone
__host__ __device__ constexpr bool scales_inside(int fmt) { return fmt == kFmtFp4 || fmt == kFmtQat || fmt == kFmtQatHp; }

// The logits S = fl32(acc c) of a column pair, rounded on their own.  The code generator contracts
// a multiply followed by an add into one fused multiply-add even when both are packed .rn
// instructions (measured: the forward's O then matched the one-rounding form bit for bit), so the
// product is formed as a fused multiply-add with a zero addend, which it leaves alone.
__device__ __forceinline__ f2 logit2(f2 a, f2 c) { return fma2(a, c, f2{0.0f, 0.0f}); }

// an fp16 pair -> the same values as a bf16 pair (exact for the fake-quantised P values)
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t *>(&b);
}

template <bool BIAS, bool MASKED, bool DUMP, int FMT, bool BF16OPS>
__device__ __forceinline__ float fwd_codes(const uint32_t (&raw)[64], float c, float rs,
                                           int nvalid, uint32_t code_col, int16_t *dump_row) {
    constexpr float kRound = 12582912.0f;          // 1.5 * 2^23
    const f2 c2{c, c}, nrs2{-rs, -rs}, rs2{rs, rs}, k127{127.0f, 127.0f}, kr2{kRound, kRound};
    const f2 k448{448.0f, 448.0f}, k2688{2688.0f, 2688.0f};
    f2 sp[2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll
    for (int cc = 0; cc < 64; cc += 16) {
        uint32_t pk[8];
        if constexpr (FMT == kFmtQat || FMT == kFmtQatHp) {
            f2 e[8];
            float emax = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                const f2 a2{__uint_as_float(raw[cc + k]), __uint_as_float(raw[cc + k + 1])};
                f2 x2 = add2(logit2(a2, c2), nrs2);            // fl32(fl32(acc c) - r)
                if (MASKED) {
                    x2.x = (cc + k < nvalid) ? x2.x : -INFINITY;
                    x2.y = (cc + k + 1 < nvalid) ? x2.y : -INFINITY;
                }
                e[k / 2] = f2{ex2_approx(x2.x), ex2_approx(x2.y)};
                sp[(k >> 1) & 1] = add2(sp[(k >> 1) & 1], e[k / 2]);
                emax = max3f(emax, e[k / 2].x, e[k / 2].y);
            }
            if constexpr (FMT == kFmtQatHp) {
#pragma unroll
                for (int k = 0; k < 8; ++k) pk[k] = BF16OPS ? pack_bf162(e[k].x, e[k].y) : pack_half2(e[k].x, e[k].y);
            } else {
                // phi: one-level NVFP4 of this 16-key group (its largest entry is at most 1)
                const float s1 = e4m3_round_f(__fdiv_rn(emax, 6.0f));
                const float inv = s1 > 0.0f ? __frcp_rn(s1) : 0.0f;
                const f2 inv2{inv, inv};
                const uint32_t s1h = pack_half2(s1, s1);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const f2 y = mul2(e[k], inv2);
                    const uint32_t h = hmul2(e2m1x2_to_f16x2(e2m1x2(y.x, y.y)), s1h);
                    pk[k] = BF16OPS ? f16x2_to_bf16x2(h) : h;
                }
            }
        } else if constexpr (FMT == kFmtFp4) {
            f2 e[8];
            float emax = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                const f2 a2{__uint_as_float(raw[cc + k]), __uint_as_float(raw[cc + k + 1])};
                f2 x2 = BIAS ? sub2(a2, rs2) : add2(logit2(a2, c2), nrs2);   // fl32(S - r), S = fl32(acc c)
                if (MASKED) {
                    x2.x = (cc + k < nvalid) ? x2.x : -INFINITY;
                    x2.y = (cc + k + 1 < nvalid) ? x2.y : -INFINITY;
                }
                e[k / 2] = f2{ex2_approx(x2.x), ex2_approx(x2.y)};
                sp[(k >> 1) & 1] = add2(sp[(k >> 1) & 1], e[k / 2]);
                emax = max3f(emax, e[k / 2].x, e[k / 2].y);
            }
            // max v = fl32(2688 max e): the rounding is monotonic
            const float s2 = e4m3_round_f(__fdiv_rn(__fmul_rn(2688.0f, emax), 6.0f));
            const float inv = s2 > 0.0f ? __frcp_rn(s2) : 0.0f;
            const f2 inv2{inv, inv};
            const uint32_t s2h = pack_half2(s2, s2);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const f2 y = mul2(mul2(k2688, e[k]), inv2);
                pk[k] = hmul2(e2m1x2_to_f16x2(e2m1x2(y.x, y.y)), s2h);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                // column pairs in packed float32 arithmetic (bit-identical to the scalar steps)
                const f2 a2{__uint_as_float(raw[cc + k]), __uint_as_float(raw[cc + k + 1])};
                f2 x2 = BIAS ? sub2(a2, rs2) : add2(logit2(a2, c2), nrs2);   // fl32(S - r), S = fl32(acc c)
                if (MASKED) {
                    x2.x = (cc + k < nvalid) ? x2.x : -INFINITY;
                    x2.y = (cc + k + 1 < nvalid) ? x2.y : -INFINITY;
                }
                const f2 e2{ex2_approx(x2.x), ex2_approx(x2.y)};
                sp[(k >> 1) & 1] = add2(sp[(k >> 1) & 1], e2);
                if (FMT == kFmtFp8) {
                    const f2 v2 = mul2(k448, e2);
                    pk[k / 2] = e4m3x2_f16x2(v2.x, v2.y);
                } else {
                    const f2 p2 = sub2(fma2(k127, e2, kr2), kr2);   // rint of the exact 127 ex2(x)
                    const float p0 = p2.x, p1 = p2.y;
                    pk[k / 2] = pack_half2(p0, p1);
                    if (DUMP && dump_row) {
                        dump_row[cc + k] = static_cast<int16_t>(p0);
                        dump_row[cc + k + 1] = static_cast<int16_t>(p1);
                    }
                }
            }
        }
        tmem_st8(code_col + cc / 2, pk);
    }
    return (sp[0].x + sp[1].x) + (sp[0].y + sp[1].y);
}

template <int D, typename OutT, bool BIAS, bool DUMP, int FMT, bool BF16OPS>
__global__ void __launch_bounds__(kThreads, 1)
sage_fwd_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, const FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // PV accumulators a tile: d = 64 fits one per 64-key half into the tile's 128 PV columns
    constexpr int kPvBuffers = D == 64 ? 2 : 1;
    const int warp = threadIdx.x >> 5;
    const int N = a.N;
    const int npair = gridDim.x;
    // causal: the longest tile pairs (the last ones) first
    const TileHead th = tile_order(a.causal);
    const int bh = th.bh;
    const int ip = a.causal ? (npair - 1 - th.rank) : th.rank;
    const int q0 = ip * 256;
    int kv_end_t[2], nsteps_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        kv_end_t[t] = tile_kv_end(q0 + 128 * t, N, a.causal);
        nsteps_t[t] = (kv_end_t[t] + 127) / 128;
    }
    const int nsteps = max(nsteps_t[0], nsteps_t[1]);
    constexpr uint32_t kTileBytes = (D / 64) * 128 * 128;

    if (warp == kMmaWarp) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        s.abort_flag = 0;
        mbar_init(&s.q_full, 1);
        for (int st = 0; st < 2; ++st) {
            mbar_init(&s.k_full[st], 1);
            mbar_init(&s.k_free[st], 1);
            mbar_init(&s.v_full[st], 1);
            mbar_init(&s.v_free[st], 1);
        }
        mbar_init(&s.mma_done, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s.s_full[t], 1);
            mbar_init(&s.p_full[t][0], 4);
            mbar_init(&s.p_full[t][1], 4);
            for (int pb = 0; pb < kPvBuffers; ++pb) {
                mbar_init(&s.pv_full[t][pb], 1);
                mbar_init(&s.pv_free[t][pb], 4);
            }
        }
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;
    if (warp >= 8) {
        regs_dec<kRegsControl>();
        if (warp == kProducerWarp) {
        // ------------------------------------------------------------------ TMA producer
        if (elect_one()) {
            tma_prefetch_desc(&mapQ);
            tma_prefetch_desc(&mapK);
            tma_prefetch_desc(&mapV);
            mbar_arrive_expect_tx(&s.q_full, 2 * kTileBytes);
            for (int t = 0; t < 2; ++t)
                for (int c = 0; c < D / 64; ++c) tma_load_3d(s.q[t][c], &mapQ, &s.q_full, 64 * c, q0 + 128 * t, bh);
            int k_issued = 0, v_issued = 0;
            // K and V tiles of step j go to stage j & 1: the next step's tiles stream in while
            // this step's MMAs still read the other stage
            for (int j = 0; j < nsteps; ++j) {
                const int st = j & 1;
                if (j >= 2 && !mbar_wait(&s.k_free[st], ((j >> 1) - 1) & 1, abort_flag, &g_fwd_err, 1)) break;
                mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c) tma_load_3d(s.k[st][c], &mapK, &s.k_full[st], 64 * c, 128 * j, bh);
                k_issued = j + 1;
                if (j >= 2 && !mbar_wait(&s.v_free[st], ((j >> 1) - 1) & 1, abort_flag, &g_fwd_err, 2)) break;
                mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c) tma_load_3d(s.v[st][c], &mapV, &s.v_full[st], 64 * c, 128 * j, bh);
                v_issued = j + 1;
            }
            // drain: every load issued must land before the CTA may exit (the last one of each
            // stage; an earlier one into the same stage was consumed before it was reissued)
            mbar_wait_drain(&s.q_full, 0, &g_fwd_err, 3);
            for (int jj = k_issued > 2 ? k_issued - 2 : 0; jj < k_issued; ++jj)
                mbar_wait_drain(&s.k_full[jj & 1], (jj >> 1) & 1, &g_fwd_err, 3);
            for (int jj = v_issued > 2 ? v_issued - 2 : 0; jj < v_issued; ++jj)
                mbar_wait_drain(&s.v_full[jj & 1], (jj >> 1) & 1, &g_fwd_err, 4);
        }
        } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        if (elect_one()) {
            constexpr uint32_t idS = idesc_f16(128, 128, BF16OPS, false, false);
            constexpr uint32_t idPV = idesc_f16(128, D, BF16OPS, false, true);
            int pv_count[2][kPvBuffers] = {};                   // [tile][PV buffer] uses
            // S_t = Q^_t K^(j)^T into the tile's S columns, K^(j) from stage kst = j & 1
            auto issue_s = [&](int t, int kst) {
                const uint32_t q_addr = smem_u32(s.q[t][0]);
                const uint32_t k_addr = smem_u32(s.k[kst][0]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                    umma_ss(tmem + 256 * t, sdesc_sw128(q_addr + off, 16, 1024),
                            sdesc_sw128(k_addr + off, 16, 1024), idS, kk > 0);
                }
                umma_commit(&s.s_full[t]);
            };
            bool ok = mbar_wait(&s.q_full, 0, abort_flag, &g_fwd_err, 5) &&
                      mbar_wait(&s.k_full[0], 0, abort_flag, &g_fwd_err, 6);
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (0 < nsteps_t[t]) issue_s(t, 0);
                umma_commit(&s.k_free[0]);
            }
            // Per step j: the PV MMAs of both tiles, half by half; a tile's S of step j + 1 goes in
            // right after its last PV of step j, so its next softmax need not wait for the other
            // tile's PVs.  That S overwrites the P codes the PV reads: this relies on the tensor pipe
            // running MMAs in issue order, which PTX guarantees only for MMAs into one accumulator.
            // Waiting for the PV to complete instead costs the forward 4 %; the outputs are
            // bit-identical either way.
            for (int j = 0; j < nsteps && ok; ++j) {
                if (!(ok = mbar_wait(&s.v_full[j & 1], (j >> 1) & 1, abort_flag, &g_fwd_err, 8))) break;
                const uint32_t v_addr = smem_u32(s.v[j & 1][0]);
                bool k_next = false;                              // K of step j + 1 has landed
                int s_left = (j + 1 < nsteps_t[0]) + (j + 1 < nsteps_t[1]);
                // half h of tile t; called with constant h and t, so that every per-tile value
                // stays in a register (indexing the small arrays at run time put them in local
                // memory, which the large shared-memory carve-out leaves to L2)
                auto pv_half = [&](const int h, const int t) -> bool {
                    if (j >= nsteps_t[t]) return true;
                    if (h == 1 && 128 * j + 64 >= kv_end_t[t]) return true;   // (then j is its last step)
                    // this half's P codes are in place (each half has its own barrier, so the
                    // first half's PV runs while the second half is being coded)
                    if (!mbar_wait(&s.p_full[t][h], j & 1, abort_flag, &g_fwd_err, 7)) return false;
                    // the PV buffer must have been read out (d = 128: the tile's one buffer, so the
                    // O update of the previous half; d = 64: this half's buffer of the last step)
                    const int pb = kPvBuffers == 2 ? h : 0;
                    if (pv_count[t][pb] > 0 &&
                        !mbar_wait(&s.pv_free[t][pb], (pv_count[t][pb] - 1) & 1, abort_flag, &g_fwd_err, 9)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t vrow = 64 * h + 16 * kk;
                        umma_ts(tmem + 256 * t + 128 + 64 * pb, tmem + 256 * t + 32 * h + 8 * kk,
                                sdesc_sw128(v_addr + vrow * 128, 16384, 1024), idPV, kk > 0);
                    }
                    umma_commit(&s.pv_full[t][pb]);
                    ++pv_count[t][pb];
                    if (h == 1 && j + 1 < nsteps_t[t]) {
                        if (!k_next) {
                            if (!mbar_wait(&s.k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_flag, &g_fwd_err, 6)) return false;
                            tc_fence_after();
                            k_next = true;
                        }
                        issue_s(t, (j + 1) & 1);
                        if (--s_left == 0) umma_commit(&s.k_free[(j + 1) & 1]);
                    }
                    return true;
                };
                ok = pv_half(0, 0) && pv_half(0, 1) && pv_half(1, 0) && pv_half(1, 1);
                if (!ok) break;
                umma_commit(&s.v_free[j & 1]);
            }
            // every MMA must have finished before the tensor memory is released
            umma_commit(&s.mma_done);
            mbar_wait_drain(&s.mma_done, 0, &g_fwd_err, 12);
        }
        }
    } else {
        regs_inc<kRegsSoftmax>();
        // ------------------------------------------------------------------ softmax warps
        const int t = warp >> 2;                      // query tile of this warpgroup
        const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
        const int row = 32 * quarter + static_cast<int>(lane_id());
        const int grow = q0 + 128 * t + row;          // query index within the head
        const int qblk = min(grow, N - 1) >> 6;
        const size_t bhN = static_cast<size_t>(bh) * N;
        const int nblk = N >> 6;
        const int kv_end = t ? kv_end_t[1] : kv_end_t[0];
        const int my_steps = t ? nsteps_t[1] : nsteps_t[0];
        // FP4: the block scales live inside the dequantised operands
        const float sq = scales_inside(FMT) ? 1.0f : a.sQ[static_cast<size_t>(bh) * nblk + qblk];
        const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 256 * t);
        float o[D];
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] = 0.0f;
        float m = -INFINITY, l = 0.0f;
        int pv_uses[kPvBuffers] = {};                 // per PV buffer
        for (int j = 0; j < my_steps; ++j) {
            if (!mbar_wait_warp(&s.s_full[t], j & 1, abort_flag, &g_fwd_err, 10)) break;
            tc_fence_after();
            const bool has_b = 128 * j + 64 < kv_end;
            float r_h0 = -INFINITY, r_h1 = -INFINITY, sum_h0 = 0.0f, sum_h1 = 0.0f;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if (h == 1 && !has_b) break;
                const int kb = 2 * j + h;                     // key block index
                const int key0 = 64 * kb;
                const float c = scales_inside(FMT) ? a.sl2
                                                   : __fmul_rn(__fmul_rn(sq, a.sK[static_cast<size_t>(bh) * nblk + kb]), a.sl2);
                // keys allowed for this row inside the block: [key0, key0 + nvalid)
                int nvalid = a.causal ? min(64, grow - key0 + 1) : 64;
                if (grow >= N) nvalid = 0;
                const float *bias = BIAS ? a.qbias + (static_cast<size_t>(bh) * nblk + qblk) * N + key0 : nullptr;
                // The 64 products of the block are read from TMEM once (four loads in flight, one
                // wait) and kept in registers for both passes.
                uint32_t raw[64];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    tmem_ld16(lane_base + 64 * h + 16 * q4, *reinterpret_cast<uint32_t(*)[16]>(&raw[16 * q4]));
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[16]>(&raw[16 * q4]));
                // pass 1: row maximum over the block (of the integer products, or of the biased
                // logits); three-input maxima take two columns per instruction
                if (DUMP) {
                    if (grow < N)
                        for (int k = 0; k < 64; ++k) a.dump_s[(bhN + grow) * N + key0 + k] = static_cast<int32_t>(__uint_as_float(raw[k]));
                }
                float r;
                if (nvalid == 64) r = fwd_row_max<BIAS, false>(raw, c, bias, 64);
                else r = fwd_row_max<BIAS, true>(raw, c, bias, nvalid);
                if (!BIAS && nvalid > 0) r = __fmul_rn(r, c);
                // Attn-QAT: the backward rebuilds this pass's P^ from r
                if (FMT == kFmtQat && grow < N) a.R[(static_cast<size_t>(bh) * nblk + kb) * N + grow] = r;
                const float rs = (r == -INFINITY) ? 0.0f : r;
                if (h == 0) r_h0 = r; else r_h1 = r;
                // pass 2: codes and the row sum; codes go to TMEM cols [32h, 32h+32) over consumed
                // S columns.  A warp with a masked column in any lane takes the masked variant.
                int16_t *dump_row = DUMP && grow < N ? a.dump_p + (bhN + grow) * N + key0 : nullptr;
                const float sum = __any_sync(0xffffffffu, nvalid < 64)
                    ? fwd_codes<BIAS, true, DUMP, FMT, BF16OPS>(raw, c, rs, nvalid, lane_base + 32 * h, dump_row)
                    : fwd_codes<BIAS, false, DUMP, FMT, BF16OPS>(raw, c, rs, 64, lane_base + 32 * h, dump_row);
                if (h == 0) sum_h0 = sum; else sum_h1 = sum;
                // this half's codes are stored: its PV MMA may start
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(&s.p_full[t][h]);
            }
            const float r_h[2] = {r_h0, r_h1}, sum_h[2] = {sum_h0, sum_h1};
            // online softmax statistics
            const float m_new = fmaxf(m, fmaxf(r_h[0], r_h[1]));
            const float alpha = (m == -INFINITY) ? 0.0f : ex2_approx(__fsub_rn(m, m_new));
            float cpv[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool live = r_h[h] != -INFINITY;
                const float g = live ? ex2_approx(__fsub_rn(r_h[h], m_new)) : 0.0f;
                l = (h == 0) ? __fmaf_rn(alpha, l, g * sum_h[h]) : __fmaf_rn(g, sum_h[h], l);
                const int kb = min(2 * j + h, nblk - 1);
                if (FMT == kFmtQat || FMT == kFmtQatHp)
                    cpv[h] = g;
                else if (FMT == kFmtFp4)
                    cpv[h] = g * (1.0f / 2688.0f);
                else
                    cpv[h] = (g * (FMT == kFmtFp8 ? 1.0f / 448.0f : 1.0f / 127.0f)) * a.sV[static_cast<size_t>(bh) * nblk + kb];
            }
            m = m_new;
            // O = alpha O + c_h PV_h
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 1 && !has_b) break;
                const int pb = kPvBuffers == 2 ? h : 0;
                if (!mbar_wait_warp(&s.pv_full[t][pb], pv_uses[pb] & 1, abort_flag, &g_fwd_err, 11)) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D; cc += 64) {
                    // 64 columns a wait, four loads in flight (32 a wait: the forward 1.2 % slower)
                    uint32_t raw[64];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld16(lane_base + 128 + 64 * pb + cc + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&raw[16 * q]));
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[16]>(&raw[16 * q]));
                    // column pairs in packed float32 arithmetic (bit-identical to the scalar steps)
#pragma unroll
                    for (int k = 0; k < 64; k += 2) {
                        const f2 pv2{__uint_as_float(raw[k]), __uint_as_float(raw[k + 1])};
                        const f2 o2{o[cc + k], o[cc + k + 1]};
                        const f2 r2 = (h == 0) ? fma2(f2{alpha, alpha}, o2, mul2(f2{cpv[0], cpv[0]}, pv2))
                                               : fma2(f2{cpv[1], cpv[1]}, pv2, o2);
                        o[cc + k] = r2.x;
                        o[cc + k + 1] = r2.y;
                    }
#pragma unroll
                    for (int k = 0; k < 64; ++k) {
                        const float pv = __uint_as_float(raw[k]);
                        if (DUMP) {
                            if (grow < N)
                                a.dump_pv[(((static_cast<size_t>(bh) * nblk + qblk) * nblk + 2 * j + h) * 64 + (grow & 63)) * D + cc + k] =
                                    static_cast<int32_t>(pv);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(&s.pv_free[t][pb]);
                ++pv_uses[pb];
            }
        }
        // epilogue: O / l in the output type, L = (m + log2 l) ln 2 (the O' pass writes O' alone)
        if (grow < N && !*abort_flag) {
            const float inv_l = 1.0f / l;
            OutT *dst = static_cast<OutT *>(a.O) + (bhN + grow) * D;
            if constexpr (std::is_same<OutT, float>::value) {
#pragma unroll
                for (int c = 0; c < D; c += 4)
                    *reinterpret_cast<float4 *>(dst + c) = make_float4(o[c] * inv_l, o[c + 1] * inv_l, o[c + 2] * inv_l, o[c + 3] * inv_l);
            } else {
#pragma unroll
            for (int c = 0; c < D; c += 8) {
                uint4 w;
                w.x = pack2<OutT>(o[c] * inv_l, o[c + 1] * inv_l);
                w.y = pack2<OutT>(o[c + 2] * inv_l, o[c + 3] * inv_l);
                w.z = pack2<OutT>(o[c + 4] * inv_l, o[c + 5] * inv_l);
                w.w = pack2<OutT>(o[c + 6] * inv_l, o[c + 7] * inv_l);
                *reinterpret_cast<uint4 *>(dst + c) = w;
            }
            }
            if (FMT != kFmtQatHp) a.L[bhN + grow] = (m + __log2f(l)) * 0.69314718055994531f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace fwd

template <int D, typename OutT, bool BIAS, bool DUMP, int FMT, bool BF16OPS = false>
static cudaError_t launch_fwd_t(const sage_params &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                const CUtensorMap &mv, const FwdArgs &a, cudaStream_t st) {
    auto kern = fwd::sage_fwd_kernel<D, OutT, BIAS, DUMP, FMT, BF16OPS>;
    const int smem = static_cast<int>(sizeof(fwd::Smem<D>)) + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the warpgroup register split must fit in what the block is launched with, or the
    // setmaxnreg increase could never be granted
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * fwd::kThreads < 2 * 128 * static_cast<int>(fwd::kRegsSoftmax) + 128 * static_cast<int>(fwd::kRegsControl))
        return cudaErrorInvalidConfiguration;
    dim3 grid((p.N + 255) / 256, p.B * p.H);
    kern<<<grid, fwd::kThreads, smem, st>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

template <int D, typename OutT>
static cudaError_t launch_fwd_d(const sage_params &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                const CUtensorMap &mv, const FwdArgs &a, cudaStream_t st) {
    using fwd::kFmtFp4;
    using fwd::kFmtFp8;
    using fwd::kFmtInt8;
    const bool bias = a.qbias != nullptr, dump = a.dump_s != nullptr;
    // the debug dump exists for the INT8 codes only (the C ABI refuses the other formats with it)
    if (a.fp4) return bias ? launch_fwd_t<D, OutT, true, false, kFmtFp4>(p, mq, mk, mv, a, st)
                           : launch_fwd_t<D, OutT, false, false, kFmtFp4>(p, mq, mk, mv, a, st);
    if (p.flags & SAGE_FLAG_FP8) return bias ? launch_fwd_t<D, OutT, true, false, kFmtFp8>(p, mq, mk, mv, a, st)
                                             : launch_fwd_t<D, OutT, false, false, kFmtFp8>(p, mq, mk, mv, a, st);
    if (dump) return bias ? launch_fwd_t<D, OutT, true, true, kFmtInt8>(p, mq, mk, mv, a, st)
                          : launch_fwd_t<D, OutT, false, true, kFmtInt8>(p, mq, mk, mv, a, st);
    return bias ? launch_fwd_t<D, OutT, true, false, kFmtInt8>(p, mq, mk, mv, a, st)
                : launch_fwd_t<D, OutT, false, false, kFmtInt8>(p, mq, mk, mv, a, st);
}

// Attn-QAT forward: both passes over the fake-quantised Q', K', V' (input 16-bit type); O and L,
// then O' (float32)
template <int D, typename T>
static cudaError_t launch_fwd_qat_d(const sage_params &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                    const CUtensorMap &mv, FwdArgs a, float *Op, cudaStream_t st) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    cudaError_t e = launch_fwd_t<D, T, false, false, fwd::kFmtQat, kBf16>(p, mq, mk, mv, a, st);
    if (e != cudaSuccess) return e;
    a.O = Op;
    return launch_fwd_t<D, float, false, false, fwd::kFmtQatHp, kBf16>(p, mq, mk, mv, a, st);
}

cudaError_t launch_fwd_qat(const sage_params &p, const void *Qf, const void *Kf, const void *Vf, FwdArgs a,
                           float *Op, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    const uint64_t bh = static_cast<uint64_t>(p.B) * p.H;
    if (!make_tmap_3d(&mq, Qf, p.d, p.N, bh) || !make_tmap_3d(&mk, Kf, p.d, p.N, bh) ||
        !make_tmap_3d(&mv, Vf, p.d, p.N, bh))
        return cudaErrorInvalidValue;
    if (p.d == 128)
        return p.dtype == SAGE_FP16 ? launch_fwd_qat_d<128, __half>(p, mq, mk, mv, a, Op, st)
                                    : launch_fwd_qat_d<128, __nv_bfloat16>(p, mq, mk, mv, a, Op, st);
    return p.dtype == SAGE_FP16 ? launch_fwd_qat_d<64, __half>(p, mq, mk, mv, a, Op, st)
                                : launch_fwd_qat_d<64, __nv_bfloat16>(p, mq, mk, mv, a, Op, st);
}

cudaError_t launch_fwd(const sage_params &p, const __half *Q16, const __half *K16,
                       const __half *V16, FwdArgs a, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    const uint64_t bh = static_cast<uint64_t>(p.B) * p.H;
    if (!make_tmap_3d(&mq, Q16, p.d, p.N, bh) || !make_tmap_3d(&mk, K16, p.d, p.N, bh) ||
        !make_tmap_3d(&mv, V16, p.d, p.N, bh))
        return cudaErrorInvalidValue;
    if (p.d == 128)
        return p.dtype == SAGE_FP16 ? launch_fwd_d<128, __half>(p, mq, mk, mv, a, st)
                                    : launch_fwd_d<128, __nv_bfloat16>(p, mq, mk, mv, a, st);
    return p.dtype == SAGE_FP16 ? launch_fwd_d<64, __half>(p, mq, mk, mv, a, st)
                                : launch_fwd_d<64, __nv_bfloat16>(p, mq, mk, mv, a, st);
}

unsigned int take_fwd_error() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_fwd_err, sizeof(v));
    cudaMemcpyToSymbol(g_fwd_err, &zero, sizeof(zero));
    return v;
}

}  // namespace sage
