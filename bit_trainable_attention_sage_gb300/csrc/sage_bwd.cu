// sage_bwd.cu -- SageBwd backward on sm_103a tensor cores (tcgen05, TMA, TMEM).
//
// Method: "SageBwd: A Trainable Low-bit Attention" (structured summary), method steps, backward
// (1)-(7); "SageAttention3 ..." (review), INT8 backward equations: D = rowsum(dO o O); recompute
// S_ij and P_ij; dV_j += MM(P^_ij^T, dO^_i) s_P s_dO; dP_ij = dO V_j^T kept in 16 bits;
// dS_ij = P_ij o (dP_ij - D_i) quantised; dQ_i += MM(dS^_ij, K^_j) s_dS s_K;
// dK_j += MM(dS^_ij^T, Q^_i) s_dS s_Q.  Section summary A.2: the backward walks key/value blocks
// and, inside, query blocks.
//
// GB300 design.  The integer GEMMs run as kind::f16 MMAs on integer-valued fp16 codes (exact, see
// the forward); dP runs on the unquantised fp16/bf16 dO and V.  One CTA owns a 128-key tile
// (two 64-key quantisation blocks) of one head and walks the head's 64-row query blocks, one
// quantisation block of queries per step.  Keys are TMEM lanes throughout:
//   S^T  = K^ Q^T   (M=128 keys, N=64 q, K=d)   } into score buffer b = step % 2, TMEM columns
//   dP^T = V dO^T   (M=128 keys, N=64 q, K=d)   } [128b, 128b+64) and [128b+64, 128b+128)
//   dK   = dS^T Q^  (M=128 keys, N=d, K=64 q; A = dS^ codes in shared memory)  -> R_B
//   dV   = P^T dO^  (M=128 keys, N=d, K=64 q; A = P codes in TMEM over S^T)   -> R_A
//   dQ   d = 128: dQ_g^T = K^_g^T dS^_g^T (M=d, N=64 q, K=64 keys of block g) -> R_B + 64 g,
//          once the dK warpgroup has read the dK product out of R_B (dK is issued first, so
//          its read-out ends first);  d = 64: dQ_g = dS^_g K^_g for two query blocks at once
//          (M=128 q, N=d) into R_Q.
// With two score buffers the tensor core computes the next block's S^T and dP^T while the score
// warpgroup turns the current block into codes, so the two overlap; a score buffer is free again
// once the dV MMA that reads its P codes has completed (the MMA thread waits for it: the tensor
// pipe's ordering covers MMAs into one accumulator only).
// Shared-memory bandwidth (128 B per clock per SM) is the bound to respect: the N = 64 MMAs read
// their A operand once per 64 queries, so nothing else goes through shared memory that need not
// (no dQ staging: dQ is reduced into global memory straight from registers).
// Warp roles (16 warps in four warpgroups):
//   warps 0-3   "score": thread = key; pass 1 reads S^T and dP^T and forms the two 64x64 tile
//               maxima (P and dS) of its key block; pass 2 reads them again, recomputes P and dS
//               bit for bit, writes P codes into TMEM (A operand of dV) and dS codes into shared
//               memory (A operand of dK, B operand of dQ).  Recomputing costs less than writing P
//               to TMEM and reading it back: TMEM traffic competes with the MMAs' accumulators.
//   warps 4-7   "dV": dV rows in registers (thread = key), scaled per product; for d = 128 it also
//               adds query rows 0-31 of each dQ product pair to global dQ (float32 reductions, a
//               warp covering 32 consecutive d of one row), for d = 64 all of dQ by vector
//               float32 reductions along each row.
//   warps 8-11  "dK": dK rows in registers; for d = 128 also dQ query rows 32-63.
//   warp 12     TMA producer: K and V once, then Q^ (3 stages), dO (2 stages), L2 / D rows (3).
//   warp 13     TMEM allocation and the single MMA-issuing thread.
//   warp 14     TMA producer of the dO^ codes (one stage).
//
// Numerics.  The method's steps are S = fl32(acc c), P = fl32(2^fl32(S - L2)) and per tile
// code = rne(fl32(x fl32(1/s))); the kernel forms fl32(acc c - L2) with one rounding, 2^x by the
// hardware approximation, and the code by rounding the exact product x * fl32(1/s), which differs
// from rne(fl32(x * inv)) only within |x * inv| 2^-24 of a half-integer.  A code can therefore
// differ from the method's only where x / s lies within rounding distance of a half-integer:
//   c = fl32(fl32(sQ sK) * fl32(log2(e)/sqrt(d)));  L2 = fl32(L * fl32(log2(e)))
//   P = fl32(ex2(fl32(acc * c - L2)))   (with Q-smoothing ex2(fl32(fl32(acc * c + bias) - L2)))
//   dS = fl32(P * fl32(dP - D))
//   per 64x64 tile: s = fl32(max|x| / 127), code = rne(x * fl32(1/s)) (the exact product rounded
//   once, codes2); max|x| < 2^-120 -> zero tile
// Attn-QAT variant ("Attn-QAT: 4-Bit Attention With Quantization-Aware Training", technical
// summary, sections 2.2-2.3): every operand is a 16-bit value of the input type -- the
// fake-quantised Q', K', V' and the plain dO (also the B operand of dV) -- and the scales are 1:
//   P  = fl32(ex2(fl32(acc c - L2))), D from the high-precision O', dS = fl32(P fl32(dP - D))
//        rounded to the input type (A operand of dK, B operand of dQ);
//   P^ = the forward's quantised P rebuilt: e = ex2(fl32(fl32(acc c) - r)) with the forward's row
//        maximum r of this (key block, query), phi(e) one-level NVFP4 over the 16 keys of a block
//        (16 lanes of a warp), P^ = rnd16(fl32(phi(e) fl32(ex2(fl32(r - L2))))) (A of dV).
// A short pass over S^T forms each 16-key block's scale once (a reduce-scatter of the block
// maxima over the lanes, one column's scale math per lane); the second pass reads S^T and dP^T.
// Nothing waits for a tile maximum, so no barrier joins the score warps.
#include "sage_device.cuh"
#include "sage_internal.h"

// Test builds only (default 0): the TMA producer never issues step 1's Q^ block, so nothing
// ever arrives on that stage's barrier and the bounded waits run out.  The library's timeout
// test builds a copy of the library with this set and a short SAGE_WAIT_CYCLES.
#ifndef SAGE_TEST_SKIP_Q_ARRIVAL
#define SAGE_TEST_SKIP_Q_ARRIVAL 0
#endif

namespace sage {

__device__ unsigned int g_bwd_err;

namespace bwd {

// Four warpgroups, launched at 128 registers a thread (512 x 128 = 65536).  setmaxnreg then gives
// score 112, dV 184, dK 184 and control 32: 128 x (112 + 184 + 184 + 32) = 65536.
constexpr int kThreads = 512;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kProducer2Warp = 14;
constexpr uint32_t kRegsScore = 112;
constexpr uint32_t kRegsDV = 184;
constexpr uint32_t kRegsDK = 184;
constexpr uint32_t kRegsControl = 32;
constexpr uint32_t kRegsLaunch = 65536 / kThreads;
static_assert(128 * (kRegsScore + kRegsDV + kRegsDK + kRegsControl) <= 65536, "register split");

// Move this warpgroup from the launch register count to R: setmaxnreg.inc may only raise the
// count and setmaxnreg.dec only lower it.
template <uint32_t R>
__device__ __forceinline__ void regs_to() {
    if constexpr (R > kRegsLaunch) regs_inc<R>();
    else if constexpr (R < kRegsLaunch) regs_dec<R>();
}
constexpr uint32_t R_A = 256;                         // dV product (d columns)
constexpr uint32_t R_B128 = R_A + 128;                // d = 128: dK product, then the dQ^T products
constexpr uint32_t R_Q = 384;                         // d = 64: the two dQ products
constexpr int kScaleSlots = 8;                        // tile scales kept for 8 steps
// operands of the dP MMA: the unquantised fp16 or bf16 dO and V (the method), or their INT8 codes
// as integer-valued fp16 (the ablation of "SageAttention3 ..." (review), Table 1c)
constexpr int kDpFp16 = 0, kDpBf16 = 1, kDpInt8 = 2;
constexpr float kTileZero = 0x1p-120f;              // tile max below which s = max / 127 is zero
constexpr float kTileZeroFp8 = 0x1p-110f;          // the same for s = max / 448 (1 / s stays finite)

template <int D>
struct Smem {
    alignas(1024) uint8_t kt[D / 64][128 * 128];       // K^ tile  [64-d chunk][key][128 B]
    alignas(1024) uint8_t vt[D / 64][128 * 128];       // V tile   (16-bit input type)
    alignas(1024) uint8_t qc[3][D / 64][64 * 128];     // Q^ blocks [stage][chunk][q][128 B]
    alignas(1024) uint8_t doc[2][D / 64][64 * 128];    // dO blocks (16-bit input type)
    alignas(1024) uint8_t dohc[D / 64][64 * 128];      // dO^ codes block
    alignas(1024) uint8_t dss[2][128 * 128];           // dS^ codes [step % 2][key][64 q], 128-byte rows
    alignas(16) float L2s[3][64];                      // [stage][q]: -fl32(L log2 e), negated
    alignas(16) float Ds[3][64];                       // [stage][q]: D
    alignas(16) float Rs[3][2][64];                    // Attn-QAT: [stage][key block][q] forward row maxima
    float4 qscal[8][64];                               // Attn-QAT: [16-key block][q] (s, 1/s, g, r)
    float red[4][2][2];                                // [warp][step parity][P max, |dS| max]
    float sps[kScaleSlots][2];                         // [step % 8][key block] P tile scales
    float sds[kScaleSlots][2];                         // [step % 8][key block] dS tile scales
    float colsum[4][128];                              // [step % 4][key] column sums of dS
    uint64_t kv_full, q_full[3], q_free[3], do_full[2], do_free[2], doh_full, doh_free;
    uint64_t meta_full[3], meta_free[3], sd_full[2], codes_ready[2];
    uint64_t a_full, a_free, b_full, b_free;           // dV product in R_A, dK product in R_B
    uint64_t aq_full, aq_free;                         // d = 128: dQ^T products in R_B
    uint64_t dv_done;                                  // the dV MMAs of a step have completed
    uint64_t rq_full, rq_free;                         // d = 64: dQ products in R_Q
    uint64_t dss_free;                                 // d = 64: the dQ MMAs are done with both dS^ tiles
    uint64_t mma_done;
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

// plain bulk copy global -> shared (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void red_add(float *addr, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// Two tile codes packed as fp16: the nearest integer (ties to even) to x * inv (inv = 0 for a zero
// tile).  fl32(x * inv + 1.5 * 2^23) rounds the exact product to an integer in one rounding (the
// float32 spacing is 1 there, and |x * inv| <= 127 * (1 + 2^-23)); the subtraction is exact and the
// integer converts to fp16 exactly.
__device__ __forceinline__ uint32_t codes2(float x0, float x1, float inv) {
    constexpr float kRound = 12582912.0f;          // 1.5 * 2^23
    const f2 y = fma2(f2{x0, x1}, f2{inv, inv}, f2{kRound, kRound});
    const f2 q = sub2(y, f2{kRound, kRound});
    return pack_half2(q.x, q.y);
}

// FP8 variant: two E4M3 tile codes e4m3(fl32(x * inv)) as fp16 values (inv = 0 for a zero tile)
__device__ __forceinline__ uint32_t codes2_e4m3(float x0, float x1, float inv) {
    const f2 y = mul2(f2{x0, x1}, f2{inv, inv});
    return e4m3x2_f16x2(y.x, y.y);
}

__device__ __forceinline__ int16_t code_lo(uint32_t w) {
    return static_cast<int16_t>(__half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))));
}
__device__ __forceinline__ int16_t code_hi(uint32_t w) {
    return static_cast<int16_t>(__half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
}

// Row data of 8 query columns (-L2 = -fl32(L log2 e) and D), loaded ahead of use: the MMAs read
// their operands from shared memory at a high rate, so a shared-memory load waited for at once
// would stall the score warps.
#ifndef SAGE_ROWDATA_LDS
#define SAGE_ROWDATA_LDS 1
#endif
struct RowData8 {
    float l2[8], dd[8];
    __device__ __forceinline__ void load(const float *L2s, const float *Ds, int col0) {
#if SAGE_ROWDATA_LDS
        // explicit shared-memory loads: through a plain pointer the compiler cannot tell the
        // address space and issues generic loads, which take the slower generic path
        const uint32_t a = smem_u32(L2s) + 4u * static_cast<uint32_t>(col0);
        const uint32_t b = smem_u32(Ds) + 4u * static_cast<uint32_t>(col0);
        *reinterpret_cast<float4 *>(&l2[0]) = lds128(a);
        *reinterpret_cast<float4 *>(&l2[4]) = lds128(a + 16u);
        *reinterpret_cast<float4 *>(&dd[0]) = lds128(b);
        *reinterpret_cast<float4 *>(&dd[4]) = lds128(b + 16u);
#else
        *reinterpret_cast<float4 *>(&l2[0]) = *reinterpret_cast<const float4 *>(&L2s[col0]);
        *reinterpret_cast<float4 *>(&l2[4]) = *reinterpret_cast<const float4 *>(&L2s[col0 + 4]);
        *reinterpret_cast<float4 *>(&dd[0]) = *reinterpret_cast<const float4 *>(&Ds[col0]);
        *reinterpret_cast<float4 *>(&dd[4]) = *reinterpret_cast<const float4 *>(&Ds[col0 + 4]);
#endif
    }
};

// P and dS of 8 query columns [col0, col0 + 8) from S^T and dP^T: P = ex2(acc c - L2) (masked to
// 0 where EDGE says the pair is not live), dS = P (dP - D).  Pass 1 and pass 2 both call this, so
// the two passes see bit-identical values.
template <bool EDGE, bool BIAS, bool DP8>
__device__ __forceinline__ void score_p_ds_8(const uint32_t (&sr)[8], const uint32_t (&dr)[8],
                                             const RowData8 &rd, int col0, float cq, float bias,
                                             int qlo, bool key_ok, float dps, float (&pv)[8],
                                             float (&ds)[8]) {
    // column pairs in packed float32 arithmetic (bit-identical to the scalar steps)
    const f2 cq2{cq, cq}, b2{bias, bias}, dps2{dps, dps};
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const f2 acc{__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])};
        const f2 l2{rd.l2[k], rd.l2[k + 1]};
        // the row data holds -L2: x = fl32(acc c - L2) is one fused multiply-add, and
        // fl32(t - L2) = fl32(t + (-L2)) exactly
        f2 x = BIAS ? add2(fma2(acc, cq2, b2), l2) : fma2(acc, cq2, l2);
        if (EDGE) {                                    // ex2(-inf) = +0: P = 0, dS = +-0
            x.x = (key_ok && col0 + k >= qlo) ? x.x : -INFINITY;
            x.y = (key_ok && col0 + k + 1 >= qlo) ? x.y : -INFINITY;
        }
        const f2 p{ex2_approx(x.x), ex2_approx(x.y)};
        // DP8: dP = fl32(integer product * fl32(s_dO s_V))
        f2 dp{__uint_as_float(dr[k]), __uint_as_float(dr[k + 1])};
        if (DP8) dp = mul2(dp, dps2);
        const f2 d = mul2(p, sub2(dp, f2{rd.dd[k], rd.dd[k + 1]}));
        pv[k] = p.x;
        pv[k + 1] = p.y;
        ds[k] = d.x;
        ds[k + 1] = d.y;
    }
}

// Walk the 64 query columns of a block 16 at a time: the TMEM loads of both 8-column halves and
// their row data go out together, one wait covers them, and the two halves are computed back to
// back, which gives the compiler eight independent column pairs to interleave.  (One 8-column
// half per wait, with the next half's loads in flight, left each wait's work too short: 2 % slower
// at d = 128 and 8 % at d = 64.  Bodies of four halves were slower still: 32 columns per wait,
// with 16 more registers for this warpgroup, by 9 % at d = 128, and 16 columns per wait with the
// next 16 columns' loads in flight (two alternating buffer sets) by 8 %.)  The loop is kept
// rolled: the four warp roles run different code on each SM sub-partition, and larger bodies
// overflow the instruction cache.
__device__ __forceinline__ void reg_fence(uint32_t (&a)[8], uint32_t (&b)[8]) {
    asm volatile("" : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
                 "+r"(a[7]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]),
                 "+r"(b[6]), "+r"(b[7]));
}
template <typename F>
__device__ __forceinline__ void score_walk(uint32_t s_col, uint32_t dp_col, const float *L2s,
                                           const float *Ds, F &&half) {
#pragma unroll 1
    for (int col0 = 0; col0 < 64; col0 += 16) {
        uint32_t sA[8], dA[8], sB[8], dB[8];
        RowData8 rA, rB;
        tmem_ld8(s_col + col0, sA);
        tmem_ld8(dp_col + col0, dA);
        tmem_ld8(s_col + col0 + 8, sB);
        tmem_ld8(dp_col + col0 + 8, dB);
        rA.load(L2s, Ds, col0);
        rB.load(L2s, Ds, col0 + 8);
        tmem_wait_ld_regs(sA, dA);
        reg_fence(sB, dB);            // (the wait covers these loads too: no use may move above it)
        half(sA, dA, rA, col0);
        half(sB, dB, rB, col0 + 8);
    }
}

// Pass 1 over the 64 query columns of a block: tile maxima of P and |dS| and the dS column sum.
template <bool EDGE, bool BIAS, bool DUMP, bool DP8>
__device__ __forceinline__ void score_pass1(uint32_t s_col, uint32_t dp_col, const float *L2s,
                                            const float *Ds, float cq, float bias, int qlo,
                                            bool key_ok, float dps, float &mp, float &md, float &cs,
                                            int32_t *dump_col0, float *dump_dp0, int N) {
    score_walk(s_col, dp_col, L2s, Ds, [&](const uint32_t(&sr)[8], const uint32_t(&dr)[8], const RowData8 &rd, int col0) {
        float pv[8], ds[8];
        score_p_ds_8<EDGE, BIAS, DP8>(sr, dr, rd, col0, cq, bias, qlo, key_ok, dps, pv, ds);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            mp = fmaxf(mp, pv[k]);
            md = fmaxf(md, fabsf(ds[k]));
            if (BIAS) cs += ds[k];
            if (DUMP && key_ok && (!EDGE || col0 + k >= qlo)) {
                dump_col0[static_cast<size_t>(col0 + k) * N] = static_cast<int32_t>(__uint_as_float(sr[k]));
                dump_dp0[static_cast<size_t>(col0 + k) * N] =
                    DP8 ? __fmul_rn(__uint_as_float(dr[k]), dps) : __uint_as_float(dr[k]);
            }
        }
    });
}

// Pass 2: P and dS recomputed from a second read of S^T and dP^T, P codes -> TMEM over S^T
// columns already read (4 packed columns at col0 / 2), dS codes -> this key's 128-byte row of the
// shared dS^ tile (16-byte chunk j stored at j ^ (key % 8), the 128-byte swizzle the MMA
// descriptors expect).
template <bool EDGE, bool BIAS, bool DUMP, bool DP8, bool FP8>
__device__ __forceinline__ void score_pass2(uint32_t s_col, uint32_t dp_col, const float *L2s,
                                            const float *Ds, float cq, float bias, int qlo,
                                            bool key_ok, float dps, float ip, float id,
                                            uint8_t *dss_row, int swz, int16_t *dump_p0,
                                            int16_t *dump_ds0, int N) {
    score_walk(s_col, dp_col, L2s, Ds, [&](const uint32_t(&sr)[8], const uint32_t(&dr)[8], const RowData8 &rd, int col0) {
        float pv[8], ds[8];
        score_p_ds_8<EDGE, BIAS, DP8>(sr, dr, rd, col0, cq, bias, qlo, key_ok, dps, pv, ds);
        uint32_t pk[4], dk[4];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            pk[k / 2] = FP8 ? codes2_e4m3(pv[k], pv[k + 1], ip) : codes2(pv[k], pv[k + 1], ip);
            dk[k / 2] = FP8 ? codes2_e4m3(ds[k], ds[k + 1], id) : codes2(ds[k], ds[k + 1], id);
            if (DUMP && key_ok) {
                dump_p0[static_cast<size_t>(col0 + k) * N] = code_lo(pk[k / 2]);
                dump_p0[static_cast<size_t>(col0 + k + 1) * N] = code_hi(pk[k / 2]);
                dump_ds0[static_cast<size_t>(col0 + k) * N] = code_lo(dk[k / 2]);
                dump_ds0[static_cast<size_t>(col0 + k + 1) * N] = code_hi(dk[k / 2]);
            }
        }
        tmem_st4(s_col + col0 / 2, pk);
        *reinterpret_cast<uint4 *>(dss_row + (((col0 >> 3) ^ swz) << 4)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
    });
}

__device__ __forceinline__ uint32_t pack16x2(float lo, float hi, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Attn-QAT pass A: the NVFP4 block data of every query column for this thread's 16-key block
// (the 16 lanes of its half-warp).  The block maximum of e = ex2(fl32(fl32(acc c) - r)) is e of the
// block maximum of acc (the float32 roundings and ex2 are monotonic), so the lanes first reduce acc:
// a reduce-scatter over the 16 lanes (offsets 8, 4, 2, 1, each step keeping half the columns)
// leaves lane L with the maxima of columns 2L and 2L + 1 of each 32-column chunk.  Each lane then
// forms, for its 4 columns, s = e4m3(fl32(max e / 6)), 1/s, g = ex2(fl32(r - L2)) and r, and stores
// them in `scal` (this half-warp's 64 columns); a column with no live key in the block gets s = 0.
template <bool EDGE>
__device__ __forceinline__ void qat_block_scales(uint32_t s_col, const float *L2s, const float *Rs,
                                                 float cq, int qlo, bool key_ok, float4 *scal) {
    const int lane = static_cast<int>(lane_id());
    const int L = lane & 15;
    float own[4];
#pragma unroll
    for (int chunk = 0; chunk < 2; ++chunk) {
        uint32_t a[32];
        tmem_ld16(s_col + 32 * chunk, *reinterpret_cast<uint32_t(*)[16]>(&a[0]));
        tmem_ld16(s_col + 32 * chunk + 16, *reinterpret_cast<uint32_t(*)[16]>(&a[16]));
        tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[16]>(&a[0]));
        tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[16]>(&a[16]));
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] = __uint_as_float(a[i]);
            if (EDGE) v[i] = (key_ok && 32 * chunk + i >= qlo) ? v[i] : -INFINITY;
        }
#pragma unroll
        for (int o = 8, w = 32; o >= 1; o >>= 1, w >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < w / 2; ++i) {
                const float send = up ? v[i] : v[i + w / 2];
                const float keep = up ? v[i + w / 2] : v[i];
                v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
            }
        }
        own[2 * chunk] = v[0];
        own[2 * chunk + 1] = v[1];
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int col = 32 * (t >> 1) + 2 * L + (t & 1);
        const float r = Rs[col];
        float sc = 0.0f, inv = 0.0f, g = 0.0f;
        if (own[t] != -INFINITY) {
            const float em = ex2_approx(__fsub_rn(__fmul_rn(own[t], cq), r));   // as the forward
            sc = e4m3_round_f(__fdiv_rn(em, 6.0f));
            inv = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
            g = ex2_approx(__fadd_rn(r, L2s[col]));     // L2s holds -L2
        }
        scal[col] = make_float4(sc, inv, g, r);
    }
    __syncwarp();
}

// Attn-QAT pass B over the 64 query columns of a block (the staging of score_walk): P and dS as
// score_p_ds_8; e = ex2(fl32(fl32(acc c) - r)) (masked to 0 where EDGE says the pair is not live);
// code = e2m1(fl32(e / s as e fl32(1/s))); P^ = rnd16(fl32((code s) g)), zero where the code is
// zero (r may be undefined for a pair the forward never visited, all of whose entries are masked).
// P^ goes to TMEM over read S^T columns, dS to this key's row of the shared dS tile.
template <bool EDGE, bool BF16>
__device__ __forceinline__ void score_pass_qat(uint32_t s_col, uint32_t dp_col, const float *L2s,
                                               const float *Ds, const float4 *scal, float cq, int qlo,
                                               bool key_ok, uint8_t *dss_row, int swz) {
    score_walk(s_col, dp_col, L2s, Ds, [&](const uint32_t(&sr)[8], const uint32_t(&dr)[8], const RowData8 &rd, int col0) {
        float pv[8], ds[8];
        score_p_ds_8<EDGE, false, false>(sr, dr, rd, col0, cq, 0.0f, qlo, key_ok, 1.0f, pv, ds);
        uint32_t pk[4], dk[4];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float4 q0 = scal[col0 + k], q1 = scal[col0 + k + 1];
            // e as the forward formed it: fl32(fl32(acc c) - r)
            float x0 = __fsub_rn(__fmul_rn(__uint_as_float(sr[k]), cq), q0.w);
            float x1 = __fsub_rn(__fmul_rn(__uint_as_float(sr[k + 1]), cq), q1.w);
            if (EDGE) {
                x0 = (key_ok && col0 + k >= qlo) ? x0 : -INFINITY;
                x1 = (key_ok && col0 + k + 1 >= qlo) ? x1 : -INFINITY;
            }
            const f2 y = mul2(f2{ex2_approx(x0), ex2_approx(x1)}, f2{q0.y, q1.y});
            const uint32_t h = e2m1x2_to_f16x2(e2m1x2(y.x, y.y));
            const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&h));
            const float p0 = c.x != 0.0f ? __fmul_rn(c.x * q0.x, q0.z) : 0.0f;   // c s is exact
            const float p1 = c.y != 0.0f ? __fmul_rn(c.y * q1.x, q1.z) : 0.0f;
            pk[k / 2] = pack16x2(p0, p1, BF16);
            dk[k / 2] = pack16x2(ds[k], ds[k + 1], BF16);
        }
        tmem_st4(s_col + col0 / 2, pk);
        *reinterpret_cast<uint4 *>(dss_row + (((col0 >> 3) ^ swz) << 4)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
    });
}

// d = 128: this warpgroup's 32 query rows [32 half, 32 half + 32) of the step's two transposed dQ
// products in R_B (thread = d column, TMEM columns = query rows): the scaled sum is added to
// global dQ by float32 reductions, one row at a time, so a warp's 32 lanes cover 32 consecutive
// floats of the row.  R_B is released once read.  (Two 8-row loads per wait: four were slower.)
// With DUMP the raw integer products of key block 0 and 1 also go to dump_g0 / dump_g1 (element
// [q][tq] of the tile's 64 x 128 product, or NULL for a key block past N).
template <bool DUMP>
__device__ __forceinline__ void dq_consume_128(uint32_t lane_base, int half, float sg0, float sg1,
                                               int tq, float *dq_rows, uint64_t *aq_free,
                                               int32_t *dump_g0, int32_t *dump_g1) {
    float *dst = dq_rows + (32 * half) * 128 + tq;
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += 8) {
        uint32_t v0[8], v1[8];
        tmem_ld8(lane_base + R_B128 + 32 * half + r0, v0);
        tmem_ld8(lane_base + R_B128 + 64 + 32 * half + r0, v1);
        tmem_wait_ld_regs(v0, v1);
        if (DUMP) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int q = 32 * half + r0 + k;
                if (dump_g0) dump_g0[q * 128] = static_cast<int32_t>(__uint_as_float(v0[k]));
                if (dump_g1) dump_g1[q * 128] = static_cast<int32_t>(__uint_as_float(v1[k]));
            }
        }
        float dq[8];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const f2 t = fma2(f2{sg1, sg1}, f2{__uint_as_float(v1[k]), __uint_as_float(v1[k + 1])},
                              mul2(f2{sg0, sg0}, f2{__uint_as_float(v0[k]), __uint_as_float(v0[k + 1])}));
            dq[k] = t.x;
            dq[k + 1] = t.y;
        }
        if (r0 + 8 == 32) {
            // every TMEM read of this warpgroup is done: R_B may be refilled
            tc_fence_before();
            __syncwarp();
            if (lane_id() == 0) mbar_arrive(aq_free);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            red_add(dst + (r0 + k) * 128, dq[k]);
    }
}

// acc[i] += sc * (product column i), i < D, from the TMEM columns [col, col + D) of this warp's
// lanes (thread = key).  Four 8-column loads share one wait: the read-out of the dV product is on
// the path to the dQ MMAs (they reuse its columns), and a wait per 8 columns left it waiting on
// TMEM latency 16 times a step (2 % of the backward call at d = 128).  With DUMP the raw integer
// products also go to dump_row (NULL for a key past N).
template <int D, bool DUMP>
__device__ __forceinline__ void add_scaled_product(uint32_t col, float sc, float (&acc)[D], int32_t *dump_row) {
#pragma unroll
    for (int cc = 0; cc < D; cc += 32) {
        uint32_t r0[8], r1[8], r2[8], r3[8];
        tmem_ld8(col + cc, r0);
        tmem_ld8(col + cc + 8, r1);
        tmem_ld8(col + cc + 16, r2);
        tmem_ld8(col + cc + 24, r3);
        tmem_wait_ld_regs(r0, r1);
        reg_fence(r2, r3);            // (the wait covers these loads too: no use may move above it)
        const uint32_t *rr[4] = {r0, r1, r2, r3};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if (DUMP && dump_row) {
#pragma unroll
                for (int k = 0; k < 8; ++k) dump_row[cc + 8 * h + k] = static_cast<int32_t>(__uint_as_float(rr[h][k]));
            }
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                const f2 t = fma2(f2{sc, sc}, f2{__uint_as_float(rr[h][k]), __uint_as_float(rr[h][k + 1])},
                                  f2{acc[cc + 8 * h + k], acc[cc + 8 * h + k + 1]});
                acc[cc + 8 * h + k] = t.x;
                acc[cc + 8 * h + k + 1] = t.y;
            }
        }
    }
}

template <int D, int DPK, bool BIAS, bool DUMP, bool QAT>
__device__ __forceinline__ void control_role(Smem<D> &s, const BwdArgs &a, const CUtensorMap *mapK, const CUtensorMap *mapV,
                                      const CUtensorMap *mapQ, const CUtensorMap *mapdO,
                                      const CUtensorMap *mapdOh) {
    const int warp = threadIdx.x >> 5;
    const int N = a.N;
    const TileHead th = tile_order(a.causal);        // causal: key tile 0, the longest, first
    const int bh = th.bh;
    const int jt = th.rank;                          // key tile: keys [128 jt, 128 jt + 128)
    const int k0 = 128 * jt;
    const int nblk = N >> 6;                         // 64-row blocks (N % 64 == 0)
    const int c_first = a.causal ? 2 * jt : 0;       // first query block with a live pair
    const int n = nblk - c_first;                    // query blocks walked (>= 1)
    const size_t bhN = static_cast<size_t>(bh) * N;
    const uint32_t tmem = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;
    (void)warp; (void)k0; (void)bhN; (void)tmem;
    constexpr uint32_t kKVBytes = (D / 64) * 128 * 128;
    constexpr uint32_t kBlkBytes = (D / 64) * 64 * 128;
    constexpr uint32_t R_B = R_A + D;
    regs_to<kRegsControl>();
    if (warp == kProducerWarp) {
        // -------------------------------------------------------------- TMA producer
        if (elect_one()) {
            tma_prefetch_desc(mapK);
            tma_prefetch_desc(mapV);
            tma_prefetch_desc(mapQ);
            tma_prefetch_desc(mapdO);
            mbar_arrive_expect_tx(&s.kv_full, 2 * kKVBytes);
            for (int c = 0; c < D / 64; ++c) {
                tma_load_3d(s.kt[c], mapK, &s.kv_full, 64 * c, k0, bh);
                tma_load_3d(s.vt[c], mapV, &s.kv_full, 64 * c, k0, bh);
            }
            int last_do[2] = {-1, -1}, last_q[3] = {-1, -1, -1}, last_meta[3] = {-1, -1, -1};
            for (int c = 0; c < n; ++c) {
                const int q0 = 64 * (c_first + c);
                const int s2 = c & 1, s3 = c % 3;
                if (c >= 2 && !mbar_wait(&s.do_free[s2], ((c >> 1) - 1) & 1, abort_flag, &g_bwd_err, 1)) break;
                mbar_arrive_expect_tx(&s.do_full[s2], kBlkBytes);
                for (int dc = 0; dc < D / 64; ++dc) tma_load_3d(s.doc[s2][dc], mapdO, &s.do_full[s2], 64 * dc, q0, bh);
                last_do[s2] = c;
                if (c >= 3 && !mbar_wait(&s.meta_free[s3], (c / 3 - 1) & 1, abort_flag, &g_bwd_err, 2)) break;
                mbar_arrive_expect_tx(&s.meta_full[s3], (QAT ? 4 : 2) * 64 * 4);
                bulk_load(s.L2s[s3], a.L2 + bhN + q0, 64 * 4, &s.meta_full[s3]);
                bulk_load(s.Ds[s3], a.D + bhN + q0, 64 * 4, &s.meta_full[s3]);
                if (QAT)
                    for (int g = 0; g < 2; ++g)
                        bulk_load(s.Rs[s3][g], a.R + (static_cast<size_t>(bh) * nblk + min(2 * jt + g, nblk - 1)) * N + q0,
                                  64 * 4, &s.meta_full[s3]);
                last_meta[s3] = c;
                if (SAGE_TEST_SKIP_Q_ARRIVAL && c == 1) continue;
                if (c >= 3 && !mbar_wait(&s.q_free[s3], (c / 3 - 1) & 1, abort_flag, &g_bwd_err, 3)) break;
                mbar_arrive_expect_tx(&s.q_full[s3], kBlkBytes);
                for (int dc = 0; dc < D / 64; ++dc) tma_load_3d(s.qc[s3][dc], mapQ, &s.q_full[s3], 64 * dc, q0, bh);
                last_q[s3] = c;
            }
            // drain: every copy issued into this CTA's shared memory has landed
            mbar_wait_drain(&s.kv_full, 0, &g_bwd_err, 4);
            for (int i = 0; i < 2; ++i)
                if (last_do[i] >= 0) mbar_wait_drain(&s.do_full[i], (last_do[i] >> 1) & 1, &g_bwd_err, 4);
            for (int i = 0; i < 3; ++i) {
                if (last_meta[i] >= 0) mbar_wait_drain(&s.meta_full[i], (last_meta[i] / 3) & 1, &g_bwd_err, 4);
                if (last_q[i] >= 0) mbar_wait_drain(&s.q_full[i], (last_q[i] / 3) & 1, &g_bwd_err, 4);
            }
        }
    } else if (warp == kProducer2Warp) {
        // -------------------------------------------------------------- dO^ producer
        if (elect_one()) {
            tma_prefetch_desc(mapdOh);
            int last = -1;
            for (int c = 0; c < n; ++c) {
                if (c >= 1 && !mbar_wait(&s.doh_free, (c - 1) & 1, abort_flag, &g_bwd_err, 5)) break;
                mbar_arrive_expect_tx(&s.doh_full, kBlkBytes);
                for (int dc = 0; dc < D / 64; ++dc)
                    tma_load_3d(s.dohc[dc], mapdOh, &s.doh_full, 64 * dc, 64 * (c_first + c), bh);
                last = c;
            }
            if (last >= 0) mbar_wait_drain(&s.doh_full, last & 1, &g_bwd_err, 4);
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        // Steady state per step c: dK(c), dV(c), dQ(c) (d = 128 into R_B once dK(c) has been read
        // out of it), then S^T / dP^T of step c + 2 into the score buffer step c used.  S^T / dP^T
        // of step c + 1 are already done, so the score warpgroup moves on at once.  The dS^ tile
        // of step c is written again at step c + 2, whose S^T / dP^T complete after dK(c) and
        // dQ(c) (d = 128), which read it; d = 64 the score warpgroup waits for dss_free.  S^T of
        // step c + 2 overwrites the P codes dV(c) reads as its A operand, and the tensor pipe's
        // ordering covers MMAs into one accumulator only, so it waits for dV(c) to complete
        // (dv_done; normally met by then: d = 128 the dK(c) read-out, d = 64 the dQ pair comes
        // in between).
        if (elect_one()) {
            // Attn-QAT: every operand in the input type; otherwise codes as fp16, dP per dtype
            constexpr bool kOpsBf16 = QAT && DPK == kDpBf16;
            constexpr uint32_t idS = idesc_f16(128, 64, kOpsBf16, false, false);   // S^T
            constexpr uint32_t idDP = idesc_f16(128, 64, DPK == kDpBf16, false, false);   // dP^T
            constexpr uint32_t idKV = idesc_f16(128, D, kOpsBf16, false, true);    // dK, dV
            constexpr uint32_t idQ = idesc_f16(128, 64, kOpsBf16, true, true);     // dQ(^T)
            // base descriptors; a byte offset `off` inside an operand adds off >> 4
            const uint64_t dKt = sdesc_sw128(smem_u32(s.kt[0]), 16, 1024);         // K-major A
            const uint64_t dVt = sdesc_sw128(smem_u32(s.vt[0]), 16, 1024);
            const uint64_t dKmn = sdesc_sw128(smem_u32(s.kt[0]), 16384, 1024);     // K^ as MN-major
            const uint64_t dDoh = sdesc_sw128(smem_u32(s.dohc[0]), 8192, 1024);    // MN-major B
            const uint64_t dDssM = sdesc_sw128(smem_u32(s.dss[0]), 16384, 1024);   // MN-major
            auto issue_sd = [&](int c) -> bool {
                const int b = c & 1, s3 = c % 3;
                if (!mbar_wait(&s.q_full[s3], (c / 3) & 1, abort_flag, &g_bwd_err, 6)) return false;
                tc_fence_after();
                const uint64_t dQk = sdesc_sw128(smem_u32(s.qc[s3][0]), 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                    umma_ss(tmem + 128 * b, dKt + oa, dQk + ob, idS, kk > 0);
                }
                if (!mbar_wait(&s.do_full[b], (c >> 1) & 1, abort_flag, &g_bwd_err, 8)) return false;
                tc_fence_after();
                const uint64_t dDo = sdesc_sw128(smem_u32(s.doc[b][0]), 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                    umma_ss(tmem + 128 * b + 64, dVt + oa, dDo + ob, idDP, kk > 0);
                }
                umma_commit(&s.sd_full[b]);
                umma_commit(&s.do_free[b]);
                return true;
            };
            bool ok = mbar_wait(&s.kv_full, 0, abort_flag, &g_bwd_err, 9);
            if (ok) ok = issue_sd(0);
            if (ok && n > 1) ok = issue_sd(1);
            for (int c = 0; c < n && ok; ++c) {
                const int b = c & 1, s3 = c % 3;
                if (!(ok = mbar_wait(&s.codes_ready[b], (c >> 1) & 1, abort_flag, &g_bwd_err, 10))) break;
                // R_B must be empty: d = 128 the dQ(c - 1) products read out, d = 64 dK(c - 1)
                if (c >= 1 && !(ok = mbar_wait(D == 128 ? &s.aq_free : &s.b_free, (c - 1) & 1, abort_flag, &g_bwd_err, 11))) break;
                tc_fence_after();
                // dK = dS^T Q^: A = this step's dS^ codes (K-major rows of 64 q), B = Q^ block
                // read as MN-major (N = d)
                {
                    const uint64_t dA = sdesc_sw128(smem_u32(s.dss[b]), 16, 1024);
                    const uint64_t dB = sdesc_sw128(smem_u32(s.qc[s3][0]), 8192, 1024);
#pragma unroll 1
                    for (int kk = 0; kk < 4; ++kk)
                        umma_ss(tmem + R_B, dA + ((kk * 32) >> 4), dB + ((kk * 2048) >> 4), idKV, kk > 0);
                }
                umma_commit(&s.b_full);
                umma_commit(&s.q_free[s3]);
                // dV = P^T dO^: A = the P codes in TMEM (8 columns per 16 q)
                if (!(ok = mbar_wait(&s.doh_full, c & 1, abort_flag, &g_bwd_err, 12))) break;
                // R_A must be empty: dV(c - 1) read out
                if (c >= 1 && !(ok = mbar_wait(&s.a_free, (c - 1) & 1, abort_flag, &g_bwd_err, 13))) break;
                tc_fence_after();
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk)
                    umma_ts(tmem + R_A, tmem + 128 * b + 8 * kk, dDoh + ((kk * 2048) >> 4), idKV, kk > 0);
                umma_commit(&s.a_full);
                umma_commit(&s.doh_free);
                umma_commit(&s.dv_done);
                if (D == 128) {
                    // dQ_g^T = K^_g^T dS^_g^T: A = K^ tile read as MN-major (M = d), B = the dS^
                    // tile read as MN-major (N = q); product g into R_B + 64 g once the dK
                    // warpgroup has read dK(c) out of R_B.  (Reusing R_A after the dV read-out,
                    // which ends one product later, made the backward 4.5 % slower: S^T / dP^T
                    // of step c + 2 queue behind dQ(c).)  dv_done first: S^T of step c + 2,
                    // issued next, overwrites dV(c)'s A operand (waiting for it after the dQ
                    // MMAs instead cost 1 %).
                    if (c + 2 < n && !(ok = mbar_wait(&s.dv_done, c & 1, abort_flag, &g_bwd_err, 17))) break;
                    if (!(ok = mbar_wait(&s.b_free, c & 1, abort_flag, &g_bwd_err, 16))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int g = 0; g < 2; ++g)
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t o = ((64 * g + 16 * kk) * 128) >> 4;
                            umma_ss(tmem + R_B + 64 * g, dKmn + o, dDssM + ((b * 16384) >> 4) + o, idQ, kk > 0);
                        }
                    umma_commit(&s.aq_full);
                } else if ((c & 1) || c == n - 1) {
                    // dQ_g = dS^_g K^_g for the step pair (c - 1, c): A = both dS^ tiles as one
                    // MN-major operand (M = 128 q), B = K^_g as MN-major (N = d)
                    const int pr = c >> 1;
                    if (pr >= 1 && !(ok = mbar_wait(&s.rq_free, (pr - 1) & 1, abort_flag, &g_bwd_err, 14))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int g = 0; g < 2; ++g)
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t o = ((64 * g + 16 * kk) * 128) >> 4;
                            umma_ss(tmem + R_Q + 64 * g, dDssM + o, dKmn + o, idQ, kk > 0);
                        }
                    umma_commit(&s.rq_full);
                    umma_commit(&s.dss_free);
                }
                if (c + 2 < n) {
                    if (D != 128 && !(ok = mbar_wait(&s.dv_done, c & 1, abort_flag, &g_bwd_err, 17))) break;
                    if (!(ok = issue_sd(c + 2))) break;
                }
            }
            umma_commit(&s.mma_done);
            mbar_wait_drain(&s.mma_done, 0, &g_bwd_err, 15);
        }
    }
}

// Score warpgroup (warps 0-3).
template <int D, int DPK, bool BIAS, bool DUMP, bool FP8, bool QAT>
__device__ __forceinline__ void score_role(Smem<D> &s, const BwdArgs &a) {
    const int warp = threadIdx.x >> 5;
    const int N = a.N;
    const TileHead th = tile_order(a.causal);        // causal: key tile 0, the longest, first
    const int bh = th.bh;
    const int jt = th.rank;                          // key tile: keys [128 jt, 128 jt + 128)
    const int k0 = 128 * jt;
    const int nblk = N >> 6;                         // 64-row blocks (N % 64 == 0)
    const int c_first = a.causal ? 2 * jt : 0;       // first query block with a live pair
    const int n = nblk - c_first;                    // query blocks walked (>= 1)
    const size_t bhN = static_cast<size_t>(bh) * N;
    const uint32_t tmem = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;
    (void)warp; (void)k0; (void)bhN; (void)tmem;
    regs_to<kRegsScore>();
    // ------------------------------------------------------------------ score warpgroup
    const int tq = threadIdx.x;                       // key lane
    const int quarter = warp;
    const int key = k0 + tq;
    const int kb = tq >> 6;
    const bool key_ok = key < N;
    const int kblk = min(2 * jt + kb, nblk - 1);
    const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
    if constexpr (QAT) {
        for (int c = 0; c < n; ++c) {
            const int q0 = 64 * (c_first + c);
            const int b = c & 1, m3 = c % 3;
            const int qlo = a.causal ? max(0, key - q0) : 0;
            const bool edge = (a.causal && q0 < k0 + 128) || k0 + 128 > N;
            if (!mbar_wait_warp(&s.meta_full[m3], (c / 3) & 1, abort_flag, &g_bwd_err, 19)) break;
            if (!mbar_wait_warp(&s.sd_full[b], (c >> 1) & 1, abort_flag, &g_bwd_err, 20)) break;
            tc_fence_after();
            if (D != 128 && c >= 2 && !mbar_wait_warp(&s.dss_free, ((c >> 1) - 1) & 1, abort_flag, &g_bwd_err, 22)) break;
            const uint32_t s_col = lane_base + 128 * b;
            uint8_t *dss_row = s.dss[b] + tq * 128;
            float4 *scal = s.qscal[tq >> 4];
            if (edge) {
                qat_block_scales<true>(s_col, s.L2s[m3], s.Rs[m3][kb], a.sl2, qlo, key_ok, scal);
                score_pass_qat<true, DPK == kDpBf16>(s_col, s_col + 64, s.L2s[m3], s.Ds[m3], scal, a.sl2, qlo,
                                                     key_ok, dss_row, tq & 7);
            } else {
                qat_block_scales<false>(s_col, s.L2s[m3], s.Rs[m3][kb], a.sl2, qlo, key_ok, scal);
                score_pass_qat<false, DPK == kDpBf16>(s_col, s_col + 64, s.L2s[m3], s.Ds[m3], scal, a.sl2, qlo,
                                                      key_ok, dss_row, tq & 7);
            }
            tmem_wait_st();
            fence_view_async_shared();
            tc_fence_before();
            __syncwarp();
            if (lane_id() == 0) {
                mbar_arrive(&s.codes_ready[b]);
                mbar_arrive(&s.meta_free[m3]);
            }
        }
        return;
    }
    const float sk = key_ok ? a.sK[static_cast<size_t>(bh) * nblk + kblk] : 0.0f;
    const float *sQh = a.sQ + static_cast<size_t>(bh) * nblk;
    const float *biash = BIAS ? a.qbias + static_cast<size_t>(bh) * nblk * N + min(key, N - 1) : nullptr;
    float sq_next = sQh[c_first];
    float b_next = (BIAS && key_ok) ? biash[static_cast<size_t>(c_first) * N] : 0.0f;
    // INT8 dP (ablation): the tile scale fl32(s_dO s_V) of the integer dP product
    const float *sdOh = a.sdO + static_cast<size_t>(bh) * nblk;
    const float sv = (DPK == kDpInt8 && key_ok) ? a.sV[static_cast<size_t>(bh) * nblk + kblk] : 0.0f;
    float sdo_next = DPK == kDpInt8 ? sdOh[c_first] : 0.0f;
    for (int c = 0; c < n; ++c) {
        const int qb = c_first + c;
        const int q0 = 64 * qb;
        const int b = c & 1, m3 = c % 3, z = c & (kScaleSlots - 1);
        const float cq = __fmul_rn(__fmul_rn(sq_next, sk), a.sl2);
        const float bias = b_next;
        const float dps = DPK == kDpInt8 ? __fmul_rn(sdo_next, sv) : 1.0f;
        if (c + 1 < n) {
            sq_next = sQh[qb + 1];
            if (BIAS && key_ok) b_next = biash[static_cast<size_t>(qb + 1) * N];
            if (DPK == kDpInt8) sdo_next = sdOh[qb + 1];
        }
        const int qlo = a.causal ? max(0, key - q0) : 0;
        const bool edge = (a.causal && q0 < k0 + 128) || k0 + 128 > N;
        // A warp whose wait gave up still takes part in this step's tile-maximum barrier, with a
        // negative maximum as its flag (P maxima are never negative): after the barrier all four
        // warps read the same four slots and leave the loop together.  A warp leaving alone would
        // leave the others blocked at the barrier.  (The give-up path is a branch of its own, so
        // that the common path keeps its register allocation.)
        if (!mbar_wait_warp(&s.meta_full[m3], (c / 3) & 1, abort_flag, &g_bwd_err, 19) ||
            !mbar_wait_warp(&s.sd_full[b], (c >> 1) & 1, abort_flag, &g_bwd_err, 20)) {
            if (lane_id() == 0) s.red[warp][c & 1][0] = -1.0f;
            named_bar_sync(1, 128);
            break;
        }
        tc_fence_after();
        const uint32_t s_col = lane_base + 128 * b;
        float mp = 0.0f, md = 0.0f, cs = 0.0f;
        int32_t *dump_s0 = DUMP ? a.dump_s + (bhN + q0) * N + key : nullptr;
        float *dump_dp0 = DUMP ? a.dump_dp + (bhN + q0) * N + key : nullptr;
        if (edge)
            score_pass1<true, BIAS, DUMP, DPK == kDpInt8>(s_col, s_col + 64, s.L2s[m3], s.Ds[m3], cq, bias, qlo,
                                                          key_ok, dps, mp, md, cs, dump_s0, dump_dp0, N);
        else
            score_pass1<false, BIAS, DUMP, DPK == kDpInt8>(s_col, s_col + 64, s.L2s[m3], s.Ds[m3], cq, bias, qlo,
                                                           key_ok, dps, mp, md, cs, dump_s0, dump_dp0, N);
        // tile maxima of (this query block, this key block): over the 32 lanes, then over the
        // two warps of the key block.  Both are non-negative floats (P >= +0, |dS|), whose bit
        // patterns order as unsigned integers: one warp-wide integer max each.
        mp = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mp)));
        md = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(md)));
        if (lane_id() == 0) {
            s.red[warp][c & 1][0] = mp;
            s.red[warp][c & 1][1] = md;
        }
        if (BIAS) s.colsum[c & 3][tq] = cs;
        named_bar_sync(1, 128);
        // a slot [w][c & 1] is written again only at step c + 2, after every warp has passed the
        // barrier of step c + 1 and so has read it here
        const float f0 = s.red[0][c & 1][0], f1 = s.red[1][c & 1][0];
        const float f2 = s.red[2][c & 1][0], f3 = s.red[3][c & 1][0];
        if (fminf(fminf(f0, f1), fminf(f2, f3)) < 0.0f) break;
        const int w0 = warp & ~1;
        const float mxp = w0 == 0 ? fmaxf(f0, f1) : fmaxf(f2, f3);
        const float mxd = fmaxf(s.red[w0][c & 1][1], s.red[w0 + 1][c & 1][1]);
        // FP8: s = max/448, and a tile below 2^-110 is zero so that 1/s stays finite
        constexpr float kZero = FP8 ? kTileZeroFp8 : kTileZero;
        constexpr float kQmax = FP8 ? 448.0f : 127.0f;
        const float sp = mxp < kZero ? 0.0f : __fdiv_rn(mxp, kQmax);
        const float ip = mxp < kZero ? 0.0f : __frcp_rn(sp);
        const float sd = mxd < kZero ? 0.0f : __fdiv_rn(mxd, kQmax);
        const float id = mxd < kZero ? 0.0f : __frcp_rn(sd);
        if ((tq & 63) == 0) {
            s.sps[z][kb] = sp;
            s.sds[z][kb] = sd;
            if (DUMP && key_ok) {
                const size_t ti = (static_cast<size_t>(bh) * nblk + qb) * nblk + kblk;
                a.dump_sp[ti] = sp;
                a.dump_sds[ti] = sd;
            }
        }
        // the dQ MMAs that read this dS^ tile two steps ago must be done: d = 128 they ran before
        // this step's S^T / dP^T (whose commit tracks every MMA issued before), d = 64 they are those of
        // the previous step pair
        // (a warp giving up here skips pass 2 and, unless this was the last step, flags the next
        // step's barrier at once: every warp has passed this step's barrier, so none still reads
        // that step's slots, and every warp reaches the next one)
        if (D != 128 && c >= 2 && !mbar_wait_warp(&s.dss_free, ((c >> 1) - 1) & 1, abort_flag, &g_bwd_err, 22)) {
            if (c + 1 < n) {
                if (lane_id() == 0) s.red[warp][(c + 1) & 1][0] = -1.0f;
                named_bar_sync(1, 128);
            }
            break;
        }
        int16_t *dump_p0 = DUMP ? a.dump_p + (bhN + q0) * N + key : nullptr;
        int16_t *dump_ds0 = DUMP ? a.dump_ds + (bhN + q0) * N + key : nullptr;
        uint8_t *dss_row = s.dss[b] + tq * 128;
        if (edge)
            score_pass2<true, BIAS, DUMP, DPK == kDpInt8, FP8>(s_col, s_col + 64, s.L2s[m3], s.Ds[m3], cq, bias, qlo, key_ok,
                                                          dps, ip, id, dss_row, tq & 7, dump_p0, dump_ds0, N);
        else
            score_pass2<false, BIAS, DUMP, DPK == kDpInt8, FP8>(s_col, s_col + 64, s.L2s[m3], s.Ds[m3], cq, bias, qlo, key_ok,
                                                           dps, ip, id, dss_row, tq & 7, dump_p0, dump_ds0, N);
        tmem_wait_st();
        fence_view_async_shared();
        tc_fence_before();
        __syncwarp();
        if (lane_id() == 0) {
            mbar_arrive(&s.codes_ready[b]);
            mbar_arrive(&s.meta_free[m3]);
        }
    }
}

// dV warpgroup (warps 4-7).
template <int D, int DPK, bool BIAS, bool DUMP, bool QAT>
__device__ __forceinline__ void dv_role(Smem<D> &s, const BwdArgs &a) {
    const int warp = threadIdx.x >> 5;
    const int N = a.N;
    const TileHead th = tile_order(a.causal);        // causal: key tile 0, the longest, first
    const int bh = th.bh;
    const int jt = th.rank;                          // key tile: keys [128 jt, 128 jt + 128)
    const int k0 = 128 * jt;
    const int nblk = N >> 6;                         // 64-row blocks (N % 64 == 0)
    const int c_first = a.causal ? 2 * jt : 0;       // first query block with a live pair
    const int n = nblk - c_first;                    // query blocks walked (>= 1)
    const size_t bhN = static_cast<size_t>(bh) * N;
    const uint32_t tmem = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;
    (void)warp; (void)k0; (void)bhN; (void)tmem;
    regs_to<kRegsDV>();
    // ------------------------------------------------------------------ dV warpgroup
    const int tq = threadIdx.x - 128;
    const int quarter = warp & 3;
    const int key = k0 + tq;
    const int kb = tq >> 6;
    const bool key_ok = key < N;
    const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
    float dv[D];
#pragma unroll
    for (int i = 0; i < D; ++i) dv[i] = 0.0f;
    float skb[2];
#pragma unroll
    for (int g = 0; g < 2; ++g)
        skb[g] = QAT ? 1.0f : (k0 + 64 * g < N) ? a.sK[static_cast<size_t>(bh) * nblk + min(2 * jt + g, nblk - 1)] : 0.0f;
    const float *sdOh = QAT ? nullptr : a.sdO + static_cast<size_t>(bh) * nblk;
    float sdo_next = QAT ? 1.0f : sdOh[c_first];
    for (int c = 0; c < n; ++c) {
        const int qb = c_first + c;
        const int q0 = 64 * qb;
        const int z = c & (kScaleSlots - 1);
        const float sdo = sdo_next;
        if (!QAT && c + 1 < n) sdo_next = sdOh[qb + 1];
        // dV += s_P s_dO (P^T dO^)
        if (!mbar_wait_warp(&s.a_full, c & 1, abort_flag, &g_bwd_err, 23)) break;
        tc_fence_after();
        {
            const float sc = QAT ? 1.0f : __fmul_rn(s.sps[z][kb], sdo);
            int32_t *dump_row = (DUMP && key_ok)
                ? a.dump_dv + (((static_cast<size_t>(bh) * nblk + qb) * nblk + 2 * jt + kb) * 64 + (tq & 63)) * D
                : nullptr;
            add_scaled_product<D, DUMP>(lane_base + R_A, sc, dv, dump_row);
        }
        tc_fence_before();
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&s.a_free);
        if (D == 128) {
            // dQ rows 0-31 of this step: both key blocks' products, each scaled by its own
            // s_dS s_K / sqrt(d), summed
            if (!mbar_wait_warp(&s.aq_full, c & 1, abort_flag, &g_bwd_err, 24)) break;
            tc_fence_after();
            const float sg0 = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[z][0], skb[0]), a.inv_sqrt_d);
            const float sg1 = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[z][1], skb[1]), a.inv_sqrt_d);
            int32_t *dq0 = nullptr, *dq1 = nullptr;
            if (DUMP) {
                const size_t t0 = (static_cast<size_t>(bh) * nblk + qb) * nblk + 2 * jt;
                if (k0 < N) dq0 = a.dump_dq + t0 * 64 * D + tq;
                if (k0 + 64 < N) dq1 = a.dump_dq + (t0 + 1) * 64 * D + tq;
            }
            dq_consume_128<DUMP>(lane_base, 0, sg0, sg1, tq, a.dQ + (bhN + q0) * D, &s.aq_free, dq0, dq1);
        } else if ((c & 1) || c == n - 1) {
            // d = 64, step pair (c - 1, c) (or the last step alone): thread = query row of the
            // pair, vector atomics along the row
            const int pr = c >> 1;
            if (!mbar_wait_warp(&s.rq_full, pr & 1, abort_flag, &g_bwd_err, 25)) break;
            tc_fence_after();
            const int zq = (2 * pr + (tq >> 6)) & (kScaleSlots - 1);
            const int qrow = 64 * (c_first + 2 * pr) + tq;
            const float s0 = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[zq][0], skb[0]), a.inv_sqrt_d);
            const float s1 = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[zq][1], skb[1]), a.inv_sqrt_d);
            const bool live = qrow < N && 2 * pr + (tq >> 6) < n;
            float *dst = a.dQ + (bhN + min(qrow, N - 1)) * D;
#pragma unroll
            for (int cc = 0; cc < 64; cc += 8) {
                uint32_t r0[8], r1[8];
                tmem_ld8(lane_base + R_Q + cc, r0);
                tmem_ld8(lane_base + R_Q + 64 + cc, r1);
                tmem_wait_ld_regs(r0, r1);
                if (DUMP && live) {
                    const size_t t0 = (static_cast<size_t>(bh) * nblk + c_first + 2 * pr + (tq >> 6)) * nblk + 2 * jt;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (k0 < N) a.dump_dq[(t0 * 64 + (tq & 63)) * D + cc + e] = static_cast<int32_t>(__uint_as_float(r0[e]));
                        if (k0 + 64 < N)
                            a.dump_dq[((t0 + 1) * 64 + (tq & 63)) * D + cc + e] = static_cast<int32_t>(__uint_as_float(r1[e]));
                    }
                }
                if (live) {
#pragma unroll
                    for (int k = 0; k < 8; k += 4) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            v[e] = __fmaf_rn(s1, __uint_as_float(r1[k + e]), __fmul_rn(s0, __uint_as_float(r0[k + e])));
                        red_add_v4(dst + cc + k, v[0], v[1], v[2], v[3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane_id() == 0) mbar_arrive(&s.rq_free);
        }
    }
    if (key_ok && !*abort_flag) {
        float *dst = a.dV + (bhN + key) * D;
#pragma unroll
        for (int i = 0; i < D; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(dv[i], dv[i + 1], dv[i + 2], dv[i + 3]);
    }
}

// dK warpgroup (warps 8-11).
template <int D, int DPK, bool BIAS, bool DUMP, bool QAT>
__device__ __forceinline__ void dk_role(Smem<D> &s, const BwdArgs &a) {
    const int warp = threadIdx.x >> 5;
    const int N = a.N;
    const TileHead th = tile_order(a.causal);        // causal: key tile 0, the longest, first
    const int bh = th.bh;
    const int jt = th.rank;                          // key tile: keys [128 jt, 128 jt + 128)
    const int k0 = 128 * jt;
    const int nblk = N >> 6;                         // 64-row blocks (N % 64 == 0)
    const int c_first = a.causal ? 2 * jt : 0;       // first query block with a live pair
    const int n = nblk - c_first;                    // query blocks walked (>= 1)
    const size_t bhN = static_cast<size_t>(bh) * N;
    const uint32_t tmem = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;
    (void)warp; (void)k0; (void)bhN; (void)tmem;
    constexpr uint32_t R_B = R_A + D;
    regs_to<kRegsDK>();
    // ------------------------------------------------------------------ dK warpgroup
    const int tq = threadIdx.x - 256;                 // key lane
    const int quarter = warp & 3;
    const int key = k0 + tq;
    const int kb = tq >> 6;
    const bool key_ok = key < N;
    const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
    float dk[D];
#pragma unroll
    for (int i = 0; i < D; ++i) dk[i] = 0.0f;
    float skb[2];
#pragma unroll
    for (int g = 0; g < 2; ++g)
        skb[g] = (k0 + 64 * g < N) ? a.sK[static_cast<size_t>(bh) * nblk + min(2 * jt + g, nblk - 1)] : 0.0f;
    const float *sQh = QAT ? nullptr : a.sQ + static_cast<size_t>(bh) * nblk;
    float sq_next = QAT ? 1.0f : sQh[c_first];
    for (int c = 0; c < n; ++c) {
        const int qb = c_first + c;
        const int q0 = 64 * qb;
        const int z = c & (kScaleSlots - 1);
        const float sq = sq_next;
        if (!QAT && c + 1 < n) sq_next = sQh[qb + 1];
        // dK += s_dS s_Q / sqrt(d) (dS^T Q^)   (+ Q-smoothing bias (dS^T 1) mu_Q / sqrt(d))
        if (!mbar_wait_warp(&s.b_full, c & 1, abort_flag, &g_bwd_err, 30)) break;
        tc_fence_after();
        {
            const float sc = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[z][kb], sq), a.inv_sqrt_d);
            int32_t *dump_row = (DUMP && key_ok)
                ? a.dump_dk + (((static_cast<size_t>(bh) * nblk + qb) * nblk + 2 * jt + kb) * 64 + (tq & 63)) * D
                : nullptr;
            add_scaled_product<D, DUMP>(lane_base + R_B, sc, dk, dump_row);
        }
        if (BIAS) {
            const float w = __fmul_rn(s.colsum[c & 3][tq], a.inv_sqrt_d);
            const float *mu = a.muQ + (static_cast<size_t>(bh) * nblk + qb) * D;
#pragma unroll
            for (int i = 0; i < D; ++i) dk[i] = __fmaf_rn(w, mu[i], dk[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&s.b_free);
        if (D == 128) {
            // dQ rows 32-63 of this step
            if (!mbar_wait_warp(&s.aq_full, c & 1, abort_flag, &g_bwd_err, 31)) break;
            tc_fence_after();
            const float sg0 = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[z][0], skb[0]), a.inv_sqrt_d);
            const float sg1 = QAT ? a.inv_sqrt_d : __fmul_rn(__fmul_rn(s.sds[z][1], skb[1]), a.inv_sqrt_d);
            int32_t *dq0 = nullptr, *dq1 = nullptr;
            if (DUMP) {
                const size_t t0 = (static_cast<size_t>(bh) * nblk + qb) * nblk + 2 * jt;
                if (k0 < N) dq0 = a.dump_dq + t0 * 64 * D + tq;
                if (k0 + 64 < N) dq1 = a.dump_dq + (t0 + 1) * 64 * D + tq;
            }
            dq_consume_128<DUMP>(lane_base, 1, sg0, sg1, tq, a.dQ + (bhN + q0) * D, &s.aq_free, dq0, dq1);
        }
    }
    if (key_ok && !*abort_flag) {
        float *dst = a.dK + (bhN + key) * D;
#pragma unroll
        for (int i = 0; i < D; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(dk[i], dk[i + 1], dk[i + 2], dk[i + 3]);
    }
}

template <int D, int DPK, bool BIAS, bool DUMP, bool FP8, bool QAT>
__global__ void __launch_bounds__(kThreads, 1)
sage_bwd_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapdO,
                const __grid_constant__ CUtensorMap mapdOh, const BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;

    if (warp == kMmaWarp) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        s.abort_flag = 0;
        uint64_t *one[] = {&s.kv_full, &s.q_full[0], &s.q_full[1], &s.q_full[2], &s.q_free[0],
                           &s.q_free[1], &s.q_free[2], &s.do_full[0], &s.do_full[1], &s.do_free[0],
                           &s.do_free[1], &s.doh_full, &s.doh_free, &s.meta_full[0],
                           &s.meta_full[1], &s.meta_full[2], &s.sd_full[0], &s.sd_full[1],
                           &s.a_full, &s.b_full, &s.aq_full, &s.rq_full, &s.dss_free,
                           &s.dv_done, &s.mma_done};
        for (uint64_t *b : one) mbar_init(b, 1);
        uint64_t *four[] = {&s.meta_free[0], &s.meta_free[1], &s.meta_free[2], &s.codes_ready[0],
                            &s.codes_ready[1], &s.a_free, &s.b_free, &s.rq_free};
        for (uint64_t *b : four) mbar_init(b, 4);
        mbar_init(&s.aq_free, 8);                    // both dQ-consuming warpgroups
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // each role computes its own CTA geometry: a value computed here and used by several roles
    // would have to sit in the same register in all of them, the 24-register control one included
    if (warp >= 12) {
        control_role<D, DPK, BIAS, DUMP, QAT>(s, a, &mapK, &mapV, &mapQ, &mapdO, &mapdOh);
        tc_fence_before();
        __syncthreads();
        if (warp == kMmaWarp) tmem_dealloc(s.tmem_base, 512);
    } else if (warp < 4) {
        score_role<D, DPK, BIAS, DUMP, FP8, QAT>(s, a);
        tc_fence_before();
        __syncthreads();
    } else if (warp < 8) {
        dv_role<D, DPK, BIAS, DUMP, QAT>(s, a);
        tc_fence_before();
        __syncthreads();
    } else {
        dk_role<D, DPK, BIAS, DUMP, QAT>(s, a);
        tc_fence_before();
        __syncthreads();
    }
}

}  // namespace bwd

template <int D, int DPK, bool BIAS, bool DUMP, bool FP8, bool QAT = false>
static cudaError_t launch_bwd_t(const sage_params &p, const CUtensorMap *maps, const BwdArgs &a,
                                cudaStream_t st) {
    auto kern = bwd::sage_bwd_kernel<D, DPK, BIAS, DUMP, FP8, QAT>;
    const int smem = static_cast<int>(sizeof(bwd::Smem<D>)) + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the warpgroup register split must fit in what the block is launched with, or the
    // setmaxnreg increase could never be granted
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * bwd::kThreads < 128 * static_cast<int>(bwd::kRegsScore + bwd::kRegsDV + bwd::kRegsDK + bwd::kRegsControl))
        return cudaErrorInvalidConfiguration;
    dim3 grid((p.N + 127) / 128, p.B * p.H);
    kern<<<grid, bwd::kThreads, smem, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a);
    return cudaGetLastError();
}

template <int D, int DPK>
static cudaError_t launch_bwd_d(const sage_params &p, const CUtensorMap *maps, const BwdArgs &a,
                                cudaStream_t st) {
    const bool bias = a.qbias != nullptr, dump = a.dump_s != nullptr;
    if (dump) return bias ? launch_bwd_t<D, DPK, true, true, false>(p, maps, a, st)
                          : launch_bwd_t<D, DPK, false, true, false>(p, maps, a, st);
    return bias ? launch_bwd_t<D, DPK, true, false, false>(p, maps, a, st)
                : launch_bwd_t<D, DPK, false, false, false>(p, maps, a, st);
}

// FP8 codes (the C ABI refuses them with the dump and with INT8 dP)
template <int D, int DPK>
static cudaError_t launch_bwd_fp8(const sage_params &p, const CUtensorMap *maps, const BwdArgs &a,
                                  cudaStream_t st) {
    return a.qbias != nullptr ? launch_bwd_t<D, DPK, true, false, true>(p, maps, a, st)
                              : launch_bwd_t<D, DPK, false, false, true>(p, maps, a, st);
}

template <int D>
static cudaError_t launch_bwd_k(const sage_params &p, const CUtensorMap *maps, const BwdArgs &a,
                                cudaStream_t st) {
    if (p.flags & SAGE_FLAG_FP8)
        return p.dtype == SAGE_BF16 ? launch_bwd_fp8<D, bwd::kDpBf16>(p, maps, a, st)
                                    : launch_bwd_fp8<D, bwd::kDpFp16>(p, maps, a, st);
    if (p.flags & SAGE_FLAG_DP_INT8) return launch_bwd_d<D, bwd::kDpInt8>(p, maps, a, st);
    return p.dtype == SAGE_BF16 ? launch_bwd_d<D, bwd::kDpBf16>(p, maps, a, st)
                                : launch_bwd_d<D, bwd::kDpFp16>(p, maps, a, st);
}

cudaError_t launch_bwd(const sage_params &p, const __half *Q16, const __half *K16,
                       const void *V, const void *dO, const __half *dO16, BwdArgs a,
                       cudaStream_t st) {
    // K^ and V: 128-row key tiles; Q^, dO and dO^: 64-row query blocks.  With SAGE_FLAG_DP_INT8
    // the caller passes the fp16 copies of the V and dO codes as V and dO.
    CUtensorMap maps[5];
    const uint64_t bh = static_cast<uint64_t>(p.B) * p.H;
    if (!make_tmap_3d(&maps[0], K16, p.d, p.N, bh, 128) || !make_tmap_3d(&maps[1], V, p.d, p.N, bh, 128) ||
        !make_tmap_3d(&maps[2], Q16, p.d, p.N, bh, 64) || !make_tmap_3d(&maps[3], dO, p.d, p.N, bh, 64) ||
        !make_tmap_3d(&maps[4], dO16, p.d, p.N, bh, 64))
        return cudaErrorInvalidValue;
    if (p.d == 128) return launch_bwd_k<128>(p, maps, a, st);
    return launch_bwd_k<64>(p, maps, a, st);
}

cudaError_t launch_bwd_qat(const sage_params &p, const void *Qf, const void *Kf, const void *Vf,
                           const void *dO, BwdArgs a, cudaStream_t st) {
    // K' and V': 128-row key tiles; Q', dO (for dP) and dO again (the B operand of dV): 64-row
    // query blocks
    CUtensorMap maps[5];
    const uint64_t bh = static_cast<uint64_t>(p.B) * p.H;
    if (!make_tmap_3d(&maps[0], Kf, p.d, p.N, bh, 128) || !make_tmap_3d(&maps[1], Vf, p.d, p.N, bh, 128) ||
        !make_tmap_3d(&maps[2], Qf, p.d, p.N, bh, 64) || !make_tmap_3d(&maps[3], dO, p.d, p.N, bh, 64) ||
        !make_tmap_3d(&maps[4], dO, p.d, p.N, bh, 64))
        return cudaErrorInvalidValue;
    const bool bf = p.dtype == SAGE_BF16;
    if (p.d == 128)
        return bf ? launch_bwd_t<128, bwd::kDpBf16, false, false, false, true>(p, maps, a, st)
                  : launch_bwd_t<128, bwd::kDpFp16, false, false, false, true>(p, maps, a, st);
    return bf ? launch_bwd_t<64, bwd::kDpBf16, false, false, false, true>(p, maps, a, st)
              : launch_bwd_t<64, bwd::kDpFp16, false, false, false, true>(p, maps, a, st);
}

unsigned int take_bwd_error() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v));
    cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
    return v;
}

}  // namespace sage
