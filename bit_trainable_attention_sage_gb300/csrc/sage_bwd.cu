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
// (two 64-key quantisation blocks) of one head and loops over 128-row query chunks (two 64-row
// blocks).  Everything is transposed so that keys are TMEM lanes:
//   S^T  = K^ Q^T      (M=128 keys, N=128 q, K=d)    TMEM R_S  = cols [0,128)
//   dP^T = V dO^T      (M=128 keys, N=128 q, K=d)    TMEM R_dP = cols [128,256)
//   two product slots R_A = cols [256,384), R_B = [384,512), each filled three times a chunk:
//     dK_h = dS^T_h Q^_h  (A from TMEM, K=64 q)    h = 0 -> R_A, 1 -> R_B
//     dV_h = P^T_h dO^_h  (A from TMEM, K=64 q)
//     dQ_g = dS^_g K^_g   (A from smem, K=64 keys)  g = key block; for d = 128 formed as
//            dQ_g^T = K^_g^T dS^_g^T (M = d) so that the dQ atomics are coalesced
// The MMA order per chunk is dK, dV, then the next chunk's S^T and dP^T (their regions' codes
// are consumed by then: the tensor pipe runs in issue order), then dQ: the score warpgroup starts
// on the next chunk while the dQ products are added to global memory.
// Warp roles (16 warps in four warpgroups):
//   warps 0-3   "score": thread = key; P = 2^(acc c - L2), dS = P o (dP - D) in place in TMEM,
//               per 64x64 tile max reductions, P and dS codes back into TMEM (A operands) and dS
//               codes into shared memory (A operand of dQ).  It holds no accumulator, so its
//               registers go to instruction-level parallelism over 16 columns at a time.
//   warps 4-7   "dV": dV rows in registers (thread = key); it also adds the two dQ products of
//               each chunk to global dQ: d = 128 stages their scaled sum in shared memory and
//               adds it with TMA bulk reductions (32 KB row blocks); d = 64 uses vector float32
//               atomics along each query row.
//   warps 8-11  "dK": dK rows in registers (thread = key).
//   warp 8     TMA producer (tiles, and L2 / D rows by bulk copy); warp 9 TMEM allocation and the
//              single MMA-issuing thread.
//
// Numerics (the CPU oracle mirrors these float32 steps):
//   c = fl32(fl32(sQ sK) * fl32(log2(e)/sqrt(d)));  L2 = fl32(L * fl32(log2(e)))
//   P = fl32(ex2(fl32(acc * c - L2)))   (with Q-smoothing ex2(fl32(fl32(acc * c + bias) - L2)))
//   dS = fl32(P * fl32(dP - D))
//   per 64x64 tile: s = fl32(max|x| / 127), code = rne16(fl32(x * fl32(1/s) + 1536)) - 1536;
//   max|x| < 2^-120 -> zero tile
#include "sage_device.cuh"
#include "sage_internal.h"

namespace sage {

__device__ unsigned int g_bwd_err;

namespace bwd {

// Four warpgroups, launched at 128 registers a thread (512 x 128 = 65536).  setmaxnreg then gives
// score 152, dV 168, dK 152 and control 40: 128 x (152 + 168 + 152 + 40) = 65536.
constexpr int kThreads = 512;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kRegsScore = 152;
constexpr uint32_t kRegsDV = 168;
constexpr uint32_t kRegsDK = 152;
constexpr uint32_t kRegsControl = 40;
constexpr uint32_t R_S = 0, R_DP = 128, R_A = 256, R_B = 384;
constexpr float kTileZero = 7.52316384526264e-37f;   // 2^-120

template <int D>
struct Smem {
    alignas(1024) uint8_t kt[D / 64][128 * 128];    // K^ tile   [chunk of 64 d][key][128 B]
    alignas(1024) uint8_t vt[D / 64][128 * 128];    // V tile    (16-bit input type)
    alignas(1024) uint8_t qc[D / 64][128 * 128];    // Q^ chunk  [chunk][q row][128 B]
    alignas(1024) uint8_t doc[D / 64][128 * 128];   // dO chunk  (16-bit input type)
    alignas(1024) uint8_t dohc[D / 64][128 * 128];  // dO^ chunk (codes)
    alignas(1024) uint8_t dss[2][128 * 128];        // dS^ as MN-major A: [q block][key][64 q]
    alignas(16) float L2s[2][128];                  // [chunk parity][q]: fl32(L log2 e)
    alignas(16) float Ds[2][128];                   // [chunk parity][q]: D
    float red[4][2][4];                             // [warp][chunk parity][4 maxima]
    float sds[2][2][2];                             // [chunk parity][kb][qb] dS tile scales
    float sps[2][2][2];                             // [chunk parity][kb][qb] P tile scales
    float colsum[2][128];                           // [qb][key] column sums of dS (Q-smoothing)
    uint64_t kv_full, q_full, q_free, do_full, do_free, doh_full, doh_free, meta_full[2];
    uint64_t s_full, dp_full, codes_ready, dss_free;
    // the two product slots R_A, R_B: "full" per consumer (the dK warpgroup takes dK, the dV
    // warpgroup dV and dQ), so that every waiter sees every phase of its barrier; "free" is shared
    // (the MMA thread waits for each use in turn)
    uint64_t a_full_k, a_full_v, a_free, b_full_k, b_full_v, b_free;
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

// TMA bulk reduction: global[dst .. dst+bytes) += shared[src ..] (float32 add), bulk-group tracked
__device__ __forceinline__ void bulk_reduce_add_f32(float *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// Two tile codes packed as fp16: rne16(fl32(x * inv + 1536)) - 1536 (inv = 0 for a zero tile).
// Values x * inv lie in [-127, 127], so x * inv + 1536 lies in [1024, 2048) where fp16 spacing is
// 1: the fp16 conversion rounds to an integer and the subtraction is exact.
__device__ __forceinline__ uint32_t codes2(float x0, float x1, float inv) {
    const float y0 = __fmaf_rn(x0, inv, 1536.0f), y1 = __fmaf_rn(x1, inv, 1536.0f);
    uint32_t r;
    // cvt packs its first source into the upper half; 0x6600 is 1536 in fp16
    asm("{\n\t.reg .b32 t;\n\t"
        "cvt.rn.f16x2.f32 t, %2, %1;\n\t"
        "sub.rn.f16x2 %0, t, %3;\n\t}"
        : "=r"(r)
        : "f"(y0), "f"(y1), "r"(0x66006600u));
    return r;
}

__device__ __forceinline__ int16_t code_lo(uint32_t w) {
    return static_cast<int16_t>(__half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))));
}
__device__ __forceinline__ int16_t code_hi(uint32_t w) {
    return static_cast<int16_t>(__half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
}

template <int D, bool BF16, bool BIAS, bool DUMP>
__global__ void __launch_bounds__(kThreads, 1)
sage_bwd_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapdO,
                const __grid_constant__ CUtensorMap mapdOh, const BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int N = a.N;
    const int bh = blockIdx.y;
    const int jt = blockIdx.x;                       // key tile: keys [128 jt, 128 jt + 128)
    const int k0 = 128 * jt;
    const int nchunks = (N + 127) / 128;
    const int c_first = a.causal ? jt : 0;           // query chunks [c_first, nchunks)
    const int nmine = nchunks - c_first;
    const int nblk = N >> 6;
    const size_t bhN = static_cast<size_t>(bh) * N;
    constexpr uint32_t kTileBytes = (D / 64) * 128 * 128;

    if (warp == kMmaWarp) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        s.abort_flag = 0;
        uint64_t *one[] = {&s.kv_full, &s.q_full, &s.q_free, &s.do_full, &s.do_free, &s.doh_full,
                           &s.doh_free, &s.meta_full[0], &s.meta_full[1], &s.s_full, &s.dp_full,
                           &s.dss_free, &s.a_full_k, &s.a_full_v, &s.b_full_k, &s.b_full_v,
                           &s.mma_done};
        for (uint64_t *b : one) mbar_init(b, 1);
        mbar_init(&s.codes_ready, 4);
        mbar_init(&s.a_free, 4);
        mbar_init(&s.b_free, 4);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;

    if (warp >= 12) {
        regs_dec<kRegsControl>();
        if (warp == kProducerWarp) {
            // -------------------------------------------------------------- TMA producer
            if (elect_one()) {
                tma_prefetch_desc(&mapK);
                tma_prefetch_desc(&mapV);
                tma_prefetch_desc(&mapQ);
                tma_prefetch_desc(&mapdO);
                tma_prefetch_desc(&mapdOh);
                mbar_arrive_expect_tx(&s.kv_full, 2 * kTileBytes);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_3d(s.kt[c], &mapK, &s.kv_full, 64 * c, k0, bh);
                    tma_load_3d(s.vt[c], &mapV, &s.kv_full, 64 * c, k0, bh);
                }
                int nq = 0, ndo = 0, ndoh = 0, nmeta[2] = {0, 0};
                for (int it = 0; it < nmine; ++it) {
                    const int q0 = 128 * (c_first + it);
                    const uint32_t rows = static_cast<uint32_t>(min(128, N - q0));
                    const int slot = it & 1;
                    if (it > 0 && !mbar_wait(&s.do_free, (it - 1) & 1, abort_flag, &g_bwd_err, 1)) break;
                    mbar_arrive_expect_tx(&s.do_full, kTileBytes);
                    for (int c = 0; c < D / 64; ++c) tma_load_3d(s.doc[c], &mapdO, &s.do_full, 64 * c, q0, bh);
                    ndo = it + 1;
                    // row data of the chunk: L2 = fl32(L log2 e) and D (written by the prologue)
                    mbar_arrive_expect_tx(&s.meta_full[slot], 8 * rows);
                    bulk_load(s.L2s[slot], a.L2 + bhN + q0, 4 * rows, &s.meta_full[slot]);
                    bulk_load(s.Ds[slot], a.D + bhN + q0, 4 * rows, &s.meta_full[slot]);
                    ++nmeta[slot];
                    if (it > 0 && !mbar_wait(&s.q_free, (it - 1) & 1, abort_flag, &g_bwd_err, 2)) break;
                    mbar_arrive_expect_tx(&s.q_full, kTileBytes);
                    for (int c = 0; c < D / 64; ++c) tma_load_3d(s.qc[c], &mapQ, &s.q_full, 64 * c, q0, bh);
                    nq = it + 1;
                    if (it > 0 && !mbar_wait(&s.doh_free, (it - 1) & 1, abort_flag, &g_bwd_err, 3)) break;
                    mbar_arrive_expect_tx(&s.doh_full, kTileBytes);
                    for (int c = 0; c < D / 64; ++c) tma_load_3d(s.dohc[c], &mapdOh, &s.doh_full, 64 * c, q0, bh);
                    ndoh = it + 1;
                }
                mbar_wait_drain(&s.kv_full, 0, &g_bwd_err, 4);
                if (ndo > 0) mbar_wait_drain(&s.do_full, (ndo - 1) & 1, &g_bwd_err, 4);
                for (int sl = 0; sl < 2; ++sl)
                    if (nmeta[sl] > 0) mbar_wait_drain(&s.meta_full[sl], (nmeta[sl] - 1) & 1, &g_bwd_err, 4);
                if (nq > 0) mbar_wait_drain(&s.q_full, (nq - 1) & 1, &g_bwd_err, 4);
                if (ndoh > 0) mbar_wait_drain(&s.doh_full, (ndoh - 1) & 1, &g_bwd_err, 4);
            }
        } else if (warp == kMmaWarp) {
            // -------------------------------------------------------------- MMA issuer
            // Per chunk: dK_0 -> A, dK_1 -> B (Q^ is then free for the next chunk), dV_0 -> A,
            // dV_1 -> B, the next chunk's S^T and dP^T, then dQ_0 -> A, dQ_1 -> B.  Each product
            // slot is refilled only after its consumer warpgroup has read it out.
            if (elect_one()) {
                constexpr uint32_t idKK = idesc_f16(128, 128, false, false, false);    // S^T
                constexpr uint32_t idDP = idesc_f16(128, 128, BF16, false, false);     // dP^T
                constexpr uint32_t idTS = idesc_f16(128, D, false, false, true);       // dV, dK
                constexpr uint32_t idQ = D == 128 ? idesc_f16(128, 128, false, true, true)   // dQ^T
                                                  : idesc_f16(128, D, false, true, true);    // dQ
                // base descriptors; a byte offset `off` inside an operand adds off >> 4
                const uint64_t dKt = sdesc_sw128(smem_u32(s.kt[0]), 16, 1024);
                const uint64_t dVt = sdesc_sw128(smem_u32(s.vt[0]), 16, 1024);
                const uint64_t dQc = sdesc_sw128(smem_u32(s.qc[0]), 16, 1024);
                const uint64_t dDo = sdesc_sw128(smem_u32(s.doc[0]), 16, 1024);
                const uint64_t dDoh = sdesc_sw128(smem_u32(s.dohc[0]), 16384, 1024);
                const uint64_t dQmn = sdesc_sw128(smem_u32(s.qc[0]), 16384, 1024);
                const uint64_t dKmn = sdesc_sw128(smem_u32(s.kt[0]), 16384, 1024);
                const uint64_t dDss = sdesc_sw128(smem_u32(s.dss[0]), 16384, 1024);
                int ua = 0, ub = 0;                        // products issued into each slot
                auto issue_s_dp = [&](int it) -> bool {
                    if (!mbar_wait(&s.q_full, it & 1, abort_flag, &g_bwd_err, 6)) return false;
                    tc_fence_after();
#pragma unroll 1
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        umma_ss(tmem + R_S, dKt + o, dQc + o, idKK, kk > 0);
                    }
                    umma_commit(&s.s_full);
                    if (!mbar_wait(&s.do_full, it & 1, abort_flag, &g_bwd_err, 8)) return false;
                    tc_fence_after();
#pragma unroll 1
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        umma_ss(tmem + R_DP, dVt + o, dDo + o, idDP, kk > 0);
                    }
                    umma_commit(&s.dp_full);
                    umma_commit(&s.do_free);
                    return true;
                };
                auto slot_ready = [&](bool is_a) -> bool {
                    const int u = is_a ? ua : ub;
                    if (u == 0) return true;
                    if (!mbar_wait(is_a ? &s.a_free : &s.b_free, (u - 1) & 1, abort_flag, &g_bwd_err, is_a ? 12 : 13)) return false;
                    tc_fence_after();
                    return true;
                };
                bool ok = mbar_wait(&s.kv_full, 0, abort_flag, &g_bwd_err, 5);
                if (ok && nmine > 0) ok = issue_s_dp(0);
                for (int it = 0; it < nmine && ok; ++it) {
                    if (!mbar_wait(&s.codes_ready, it & 1, abort_flag, &g_bwd_err, 10)) break;
                    tc_fence_after();
                    // dK_h = dS^T[:, h] Q^_h
#pragma unroll 1
                    for (int h = 0; h < 2 && ok; ++h) {
                        if (!(ok = slot_ready(h == 0))) break;
                        const uint32_t dst = tmem + (h == 0 ? R_A : R_B);
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ts(dst, tmem + R_DP + 32 * h + 8 * kk, dQmn + (((64 * h + 16 * kk) * 128) >> 4), idTS, kk > 0);
                        umma_commit(h == 0 ? &s.a_full_k : &s.b_full_k);
                        if (h == 0) ++ua; else ++ub;
                    }
                    if (!ok) break;
                    umma_commit(&s.q_free);
                    if (!mbar_wait(&s.doh_full, it & 1, abort_flag, &g_bwd_err, 11)) break;
                    // dV_h = P^T[:, h] dO^_h
#pragma unroll 1
                    for (int h = 0; h < 2 && ok; ++h) {
                        if (!(ok = slot_ready(h == 0))) break;
                        const uint32_t dst = tmem + (h == 0 ? R_A : R_B);
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ts(dst, tmem + R_S + 32 * h + 8 * kk, dDoh + (((64 * h + 16 * kk) * 128) >> 4), idTS, kk > 0);
                        umma_commit(h == 0 ? &s.a_full_v : &s.b_full_v);
                        if (h == 0) ++ua; else ++ub;
                    }
                    if (!ok) break;
                    umma_commit(&s.doh_free);
                    // the next chunk's scores: the tensor pipe runs in issue order, so the codes in
                    // R_S / R_DP have been read by the dV / dK MMAs above before they are replaced
                    if (it + 1 < nmine && !(ok = issue_s_dp(it + 1))) break;
                    // dQ_g = dS^[:, keys of g] K^_g.  For d = 128 it is formed transposed,
                    // dQ_g^T = K^_g^T dS^_g^T (M = d, N = 128 q): same two shared tiles with the
                    // operand roles swapped, so that a thread then owns one d column and the
                    // atomic adds of a warp hit 32 consecutive floats of one query row.
#pragma unroll 1
                    for (int g = 0; g < 2 && ok; ++g) {
                        if (!(ok = slot_ready(g == 0))) break;
                        const uint32_t dst = tmem + (g == 0 ? R_A : R_B);
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t o = ((64 * g + 16 * kk) * 128) >> 4;
                            if (D == 128) umma_ss(dst, dKmn + o, dDss + o, idQ, kk > 0);
                            else umma_ss(dst, dDss + o, dKmn + o, idQ, kk > 0);
                        }
                        umma_commit(g == 0 ? &s.a_full_v : &s.b_full_v);
                        if (g == 0) ++ua; else ++ub;
                    }
                    // d = 64: the dS^ tile is free once the dQ MMAs have read it; d = 128: the dV
                    // warpgroup frees it after staging the dQ reduction through it
                    if (D != 128) umma_commit(&s.dss_free);
                }
                umma_commit(&s.mma_done);
                mbar_wait_drain(&s.mma_done, 0, &g_bwd_err, 14);
            }
        }
    } else if (warp < 4) {
        regs_inc<kRegsScore>();
        // ------------------------------------------------------------------ score warpgroup
        const int tq = threadIdx.x;                       // 0..127: key lane
        const int quarter = warp;
        const int key = k0 + tq;                          // key index within the head
        const int kb = tq >> 6;                           // key block of this lane (0/1)
        const int kblk = min(key, N - 1) >> 6;            // global key block
        const bool key_ok = key < N;
        const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
        const float sk = a.sK[static_cast<size_t>(bh) * nblk + kblk];
        // per-chunk scalars, fetched one chunk ahead
        const float *sQh = a.sQ + static_cast<size_t>(bh) * nblk;
        const float *biash = BIAS ? a.qbias + static_cast<size_t>(bh) * nblk * N + min(key, N - 1) : nullptr;
        float sq0 = 0.0f, sq1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
        if (nmine > 0) {
            sq0 = sQh[min(2 * c_first, nblk - 1)];
            sq1 = sQh[min(2 * c_first + 1, nblk - 1)];
            if (BIAS && key_ok) {
                b0 = biash[static_cast<size_t>(min(2 * c_first, nblk - 1)) * N];
                b1 = biash[static_cast<size_t>(min(2 * c_first + 1, nblk - 1)) * N];
            }
        }
        for (int it = 0; it < nmine; ++it) {
            const uint32_t ph = it & 1;
            const int slot = it & 1;
            const int ic = c_first + it;
            const int q0 = 128 * ic;
            float nsq0 = 0.0f, nsq1 = 0.0f, nb0 = 0.0f, nb1 = 0.0f;
            if (it + 1 < nmine) {
                nsq0 = sQh[min(2 * ic + 2, nblk - 1)];
                nsq1 = sQh[min(2 * ic + 3, nblk - 1)];
                if (BIAS && key_ok) {
                    nb0 = biash[static_cast<size_t>(min(2 * ic + 2, nblk - 1)) * N];
                    nb1 = biash[static_cast<size_t>(min(2 * ic + 3, nblk - 1)) * N];
                }
            }
            const float cq[2] = {__fmul_rn(__fmul_rn(sq0, sk), a.sl2), __fmul_rn(__fmul_rn(sq1, sk), a.sl2)};
            const float biasv[2] = {b0, b1};
            // valid query columns for this key: [qlo, qhi) relative to q0
            const int qhi = min(128, N - q0);
            const int qlo = a.causal ? max(0, key - q0) : 0;
            const bool edge = (a.causal && ic == jt) || q0 + 128 > N || k0 + 128 > N;
            if (!mbar_wait(&s.meta_full[slot], (it >> 1) & 1, abort_flag, &g_bwd_err, 19)) break;
            if (!mbar_wait(&s.s_full, ph, abort_flag, &g_bwd_err, 20)) break;
            if (!mbar_wait(&s.dp_full, ph, abort_flag, &g_bwd_err, 21)) break;
            tc_fence_after();
            // pass 1: P and dS in place, tile maxima, column sums of dS
            float mp[2] = {0.0f, 0.0f}, md[2] = {0.0f, 0.0f}, cs[2] = {0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll 1
            for (int cc = 64 * h; cc < 64 * h + 64; cc += 8) {
                uint32_t sr[8], dr[8];
                tmem_ld8(lane_base + R_S + cc, sr);
                tmem_ld8(lane_base + R_DP + cc, dr);
                float l2v[8], dvv[8];
#pragma unroll
                for (int k = 0; k < 8; k += 4) {
                    *reinterpret_cast<float4 *>(&l2v[k]) = *reinterpret_cast<const float4 *>(&s.L2s[slot][cc + k]);
                    *reinterpret_cast<float4 *>(&dvv[k]) = *reinterpret_cast<const float4 *>(&s.Ds[slot][cc + k]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int col = cc + k;
                    const float acc = __uint_as_float(sr[k]);
                    float x;
                    if (BIAS) x = __fsub_rn(__fmaf_rn(acc, cq[h], biasv[h]), l2v[k]);
                    else x = __fmaf_rn(acc, cq[h], -l2v[k]);
                    float p = ex2_approx(x);
                    float ds = __fmul_rn(p, __fsub_rn(__uint_as_float(dr[k]), dvv[k]));
                    if (edge) {
                        const bool ok = key_ok && col >= qlo && col < qhi;
                        p = ok ? p : 0.0f;
                        ds = ok ? ds : 0.0f;
                        if (DUMP) {
                            if (ok) a.dump_s[(bhN + q0 + col) * N + key] = static_cast<int32_t>(acc);
                        }
                    } else if (DUMP) {
                        a.dump_s[(bhN + q0 + col) * N + key] = static_cast<int32_t>(acc);
                    }
                    mp[h] = fmaxf(mp[h], p);
                    md[h] = fmaxf(md[h], fabsf(ds));
                    if (BIAS) cs[h] += ds;
                    sr[k] = __float_as_uint(p);
                    dr[k] = __float_as_uint(ds);
                }
                tmem_st8(lane_base + R_S + cc, sr);
                tmem_st8(lane_base + R_DP + cc, dr);
            }
            tmem_wait_st();
            // per 64x64 tile maxima: over the 32 lanes, then over the two warps of this key block
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    mp[h] = fmaxf(mp[h], __shfl_xor_sync(0xffffffffu, mp[h], o));
                    md[h] = fmaxf(md[h], __shfl_xor_sync(0xffffffffu, md[h], o));
                }
            }
            if (lane_id() == 0) {
                s.red[warp][slot][0] = mp[0];
                s.red[warp][slot][1] = mp[1];
                s.red[warp][slot][2] = md[0];
                s.red[warp][slot][3] = md[1];
            }
            if (BIAS) {
                s.colsum[0][tq] = cs[0];
                s.colsum[1][tq] = cs[1];
            }
            named_bar_sync(1, 128);
            const int w0 = warp & ~1;
            float sp[2], sd[2], ip[2], id[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float mxp = fmaxf(s.red[w0][slot][h], s.red[w0 + 1][slot][h]);
                const float mxd = fmaxf(s.red[w0][slot][2 + h], s.red[w0 + 1][slot][2 + h]);
                sp[h] = mxp < kTileZero ? 0.0f : __fdiv_rn(mxp, 127.0f);
                ip[h] = mxp < kTileZero ? 0.0f : __frcp_rn(sp[h]);
                sd[h] = mxd < kTileZero ? 0.0f : __fdiv_rn(mxd, 127.0f);
                id[h] = mxd < kTileZero ? 0.0f : __frcp_rn(sd[h]);
            }
            if ((tq & 63) == 0) {
                s.sds[slot][kb][0] = sd[0];
                s.sds[slot][kb][1] = sd[1];
                s.sps[slot][kb][0] = sp[0];
                s.sps[slot][kb][1] = sp[1];
                if (DUMP) {
                    for (int h = 0; h < 2; ++h) {
                        if (key_ok && q0 + 64 * h < N) {
                            const size_t ti = (static_cast<size_t>(bh) * nblk + 2 * ic + h) * nblk + kblk;
                            a.dump_sp[ti] = sp[h];
                            a.dump_sds[ti] = sd[h];
                        }
                    }
                }
            }
            // the dQ MMAs of the previous chunk must be done with the dS^ shared tile
            if (it > 0 && !mbar_wait(&s.dss_free, (it - 1) & 1, abort_flag, &g_bwd_err, 22)) break;
            // pass 2: codes -> TMEM (P^T over R_S, dS^T over R_DP) and dS^ -> shared (MN-major A)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll 1
            for (int cc = 64 * h; cc < 64 * h + 64; cc += 16) {
                uint32_t pr[16], dr[16];
                tmem_ld16(lane_base + R_S + cc, pr);
                tmem_ld16(lane_base + R_DP + cc, dr);
                tmem_wait_ld();
                uint32_t pk[8], dk[8];
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    pk[k / 2] = codes2(__uint_as_float(pr[k]), __uint_as_float(pr[k + 1]), ip[h]);
                    dk[k / 2] = codes2(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1]), id[h]);
                    if (DUMP) {
                        const int col = cc + k;
                        if (key_ok && q0 + col < N) {
                            a.dump_p[(bhN + q0 + col) * N + key] = code_lo(pk[k / 2]);
                            a.dump_ds[(bhN + q0 + col) * N + key] = code_lo(dk[k / 2]);
                        }
                        if (key_ok && q0 + col + 1 < N) {
                            a.dump_p[(bhN + q0 + col + 1) * N + key] = code_hi(pk[k / 2]);
                            a.dump_ds[(bhN + q0 + col + 1) * N + key] = code_hi(dk[k / 2]);
                        }
                    }
                }
                tmem_st8(lane_base + R_S + cc / 2, pk);
                tmem_st8(lane_base + R_DP + cc / 2, dk);
                // dS^ row of this key, q columns [cc, cc+16) -> two 16-byte chunks of the 128-byte
                // row (q % 64) of block h, swizzled: chunk index ^= key % 8
                uint8_t *row = s.dss[h] + tq * 128;
                const int c16 = (cc & 63) >> 3;                    // first 16-byte chunk (8 q each)
                *reinterpret_cast<uint4 *>(row + (((c16) ^ (tq & 7)) << 4)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
                *reinterpret_cast<uint4 *>(row + (((c16 + 1) ^ (tq & 7)) << 4)) = make_uint4(dk[4], dk[5], dk[6], dk[7]);
            }
            tmem_wait_st();
            fence_view_async_shared();
            tc_fence_before();
            __syncwarp();
            if (lane_id() == 0) mbar_arrive(&s.codes_ready);
            sq0 = nsq0;
            sq1 = nsq1;
            b0 = nb0;
            b1 = nb1;
        }
    } else if (warp < 8) {
        regs_inc<kRegsDV>();
        // ------------------------------------------------------------------ dV warpgroup
        // dV rows in registers (thread = key); the two dQ products of each chunk (d = 128:
        // thread = d column) scaled, summed and added to global dQ with float32 atomics
        const int tq = threadIdx.x - 128;
        const int quarter = warp & 3;
        const int key = k0 + tq;
        const int kb = tq >> 6;
        const bool key_ok = key < N;
        const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
        float dv[D];
#pragma unroll
        for (int c = 0; c < D; ++c) dv[c] = 0.0f;
        float skb[2];
#pragma unroll
        for (int g = 0; g < 2; ++g)
            skb[g] = (k0 + 64 * g < N) ? a.sK[static_cast<size_t>(bh) * nblk + min(2 * jt + g, nblk - 1)] : 0.0f;
        float sdo[2], nsdo[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) sdo[h] = nmine > 0 ? a.sdO[static_cast<size_t>(bh) * nblk + min(2 * c_first + h, nblk - 1)] : 0.0f;
        for (int it = 0; it < nmine; ++it) {
            const int ic = c_first + it;
            const int q0 = 128 * ic;
            const int slot = it & 1;
            if (it + 1 < nmine) {
#pragma unroll
                for (int h = 0; h < 2; ++h) nsdo[h] = a.sdO[static_cast<size_t>(bh) * nblk + min(2 * ic + 2 + h, nblk - 1)];
            }
            // dV += s_P s_dO (P^T dO^)_h: product h in slot A (h = 0) or B (h = 1); this
            // warpgroup's barrier of a slot completes twice a chunk: dV (parity 0), then dQ (1)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!mbar_wait(h == 0 ? &s.a_full_v : &s.b_full_v, 0, abort_flag, &g_bwd_err, 23)) break;
                tc_fence_after();
                const float sc = __fmul_rn(s.sps[slot][kb][h], sdo[h]);
                const uint32_t src = lane_base + (h == 0 ? R_A : R_B);
#pragma unroll
                for (int cc = 0; cc < D; cc += 8) {
                    uint32_t r[8];
                    tmem_ld8(src + cc, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 8; ++k) dv[cc + k] = __fmaf_rn(sc, __uint_as_float(r[k]), dv[cc + k]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(h == 0 ? &s.a_free : &s.b_free);
            }
            // dQ: both key blocks' products, each scaled by its own s_dS s_K / sqrt(d) and summed
            if (!mbar_wait(&s.a_full_v, 1, abort_flag, &g_bwd_err, 31)) break;
            if (!mbar_wait(&s.b_full_v, 1, abort_flag, &g_bwd_err, 32)) break;
            tc_fence_after();
            if (D == 128) {
                // transposed products: thread = d column c, TMEM columns = the chunk's query rows.
                // The scaled sum goes to shared memory (the dS^ tile, which the dQ MMAs have
                // finished reading) as 64 query rows x 128 floats at a time, and one TMA bulk
                // reduction adds each 32 KB block of rows to global dQ.
                const int c = tq;
                float sg0[2], sg1[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    sg0[h] = __fmul_rn(__fmul_rn(s.sds[slot][0][h], skb[0]), a.inv_sqrt_d);
                    sg1[h] = __fmul_rn(__fmul_rn(s.sds[slot][1][h], skb[1]), a.inv_sqrt_d);
                }
                const int nrow = min(128, N - q0);
                float *stage = reinterpret_cast<float *>(s.dss[0]);        // [64 rows][128 floats]
                const bool leader = tq == 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int rows = min(64, nrow - 64 * h);
                    if (rows <= 0) break;
                    if (h == 1) {
                        // the first block's reduction must have read the staging tile
                        if (leader) bulk_wait_read_all();
                        named_bar_sync(2, 128);
                    }
#pragma unroll 1
                    for (int cc = 64 * h; cc < 64 * h + 64; cc += 8) {
                        uint32_t r0[8], r1[8];
                        tmem_ld8(lane_base + R_A + cc, r0);
                        tmem_ld8(lane_base + R_B + cc, r1);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            stage[(cc - 64 * h + k) * 128 + c] =
                                __fmaf_rn(sg1[h], __uint_as_float(r1[k]), __fmul_rn(sg0[h], __uint_as_float(r0[k])));
                    }
                    fence_view_async_shared();
                    named_bar_sync(2, 128);
                    if (leader) {
                        bulk_reduce_add_f32(a.dQ + (bhN + q0 + 64 * h) * D, stage, static_cast<uint32_t>(rows) * 128u * 4u);
                        bulk_commit();
                    }
                }
                // the products have been read out of TMEM: release both slots
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) {
                    mbar_arrive(&s.a_free);
                    mbar_arrive(&s.b_free);
                }
                // the staging tile goes back to the score warpgroup once the last reduction read it
                if (leader) {
                    bulk_wait_read_all();
                    mbar_arrive(&s.dss_free);
                }
            } else {
                // d = 64: thread = query row of the chunk, vector atomics along the row
                const int qrow = q0 + tq;
                const int h_row = tq >> 6;
                const float s0 = __fmul_rn(__fmul_rn(s.sds[slot][0][h_row], skb[0]), a.inv_sqrt_d);
                const float s1 = __fmul_rn(__fmul_rn(s.sds[slot][1][h_row], skb[1]), a.inv_sqrt_d);
                const bool live = qrow < N;
                float *dst = a.dQ + (bhN + min(qrow, N - 1)) * D;
#pragma unroll 1
                for (int cc = 0; cc < D; cc += 8) {
                    uint32_t r0[8], r1[8];
                    tmem_ld8(lane_base + R_A + cc, r0);
                    tmem_ld8(lane_base + R_B + cc, r1);
                    tmem_wait_ld();
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
            }
            if (D != 128) {
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) {
                    mbar_arrive(&s.a_free);
                    mbar_arrive(&s.b_free);
                }
            }
            if (it + 1 < nmine) {
#pragma unroll
                for (int h = 0; h < 2; ++h) sdo[h] = nsdo[h];
            }
        }
        if (D == 128 && tq == 0) bulk_wait_all();
        if (key_ok && !*abort_flag) {
            float *dst = a.dV + (bhN + key) * D;
#pragma unroll
            for (int c = 0; c < D; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(dv[c], dv[c + 1], dv[c + 2], dv[c + 3]);
        }
    } else {
        regs_inc<kRegsDK>();
        // ------------------------------------------------------------------ dK warpgroup
        const int tq = threadIdx.x - 256;                 // key lane
        const int quarter = warp & 3;
        const int key = k0 + tq;
        const int kb = tq >> 6;
        const bool key_ok = key < N;
        const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
        float dk[D];
#pragma unroll
        for (int c = 0; c < D; ++c) dk[c] = 0.0f;
        float skb[2];
#pragma unroll
        for (int g = 0; g < 2; ++g)
            skb[g] = (k0 + 64 * g < N) ? a.sK[static_cast<size_t>(bh) * nblk + min(2 * jt + g, nblk - 1)] : 0.0f;
        float sq[2], nsq[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) sq[h] = nmine > 0 ? a.sQ[static_cast<size_t>(bh) * nblk + min(2 * c_first + h, nblk - 1)] : 0.0f;
        for (int it = 0; it < nmine; ++it) {
            const int ic = c_first + it;
            const int q0 = 128 * ic;
            const int slot = it & 1;
            if (it + 1 < nmine) {
#pragma unroll
                for (int h = 0; h < 2; ++h) nsq[h] = a.sQ[static_cast<size_t>(bh) * nblk + min(2 * ic + 2 + h, nblk - 1)];
            }
            // dK += s_dS s_Q / sqrt(d) (dS^T Q^)_h   (+ Q-smoothing bias (dS^T 1) mu_Q / sqrt(d));
            // this warpgroup's barrier of a slot completes once a chunk
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!mbar_wait(h == 0 ? &s.a_full_k : &s.b_full_k, it & 1, abort_flag, &g_bwd_err, 30)) break;
                tc_fence_after();
                const float sc = __fmul_rn(__fmul_rn(s.sds[slot][kb][h], sq[h]), a.inv_sqrt_d);
                const uint32_t src = lane_base + (h == 0 ? R_A : R_B);
#pragma unroll
                for (int cc = 0; cc < D; cc += 8) {
                    uint32_t r[8];
                    tmem_ld8(src + cc, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 8; ++k) dk[cc + k] = __fmaf_rn(sc, __uint_as_float(r[k]), dk[cc + k]);
                }
                if (BIAS && q0 + 64 * h < N) {
                    const float w = __fmul_rn(s.colsum[h][tq], a.inv_sqrt_d);
                    const float *mu = a.muQ + (static_cast<size_t>(bh) * nblk + min(2 * ic + h, nblk - 1)) * D;
#pragma unroll
                    for (int c = 0; c < D; ++c) dk[c] = __fmaf_rn(w, mu[c], dk[c]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(h == 0 ? &s.a_free : &s.b_free);
            }
            if (it + 1 < nmine) {
#pragma unroll
                for (int h = 0; h < 2; ++h) sq[h] = nsq[h];
            }
        }
        if (key_ok && !*abort_flag) {
            float *dst = a.dK + (bhN + key) * D;
#pragma unroll
            for (int c = 0; c < D; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(dk[c], dk[c + 1], dk[c + 2], dk[c + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace bwd

template <int D, bool BF16, bool BIAS, bool DUMP>
static cudaError_t launch_bwd_t(const sage_params &p, const CUtensorMap *maps, const BwdArgs &a,
                                cudaStream_t st) {
    auto kern = bwd::sage_bwd_kernel<D, BF16, BIAS, DUMP>;
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

template <int D, bool BF16>
static cudaError_t launch_bwd_d(const sage_params &p, const CUtensorMap *maps, const BwdArgs &a,
                                cudaStream_t st) {
    const bool bias = a.qbias != nullptr, dump = a.dump_s != nullptr;
    if (dump) return bias ? launch_bwd_t<D, BF16, true, true>(p, maps, a, st)
                          : launch_bwd_t<D, BF16, false, true>(p, maps, a, st);
    return bias ? launch_bwd_t<D, BF16, true, false>(p, maps, a, st)
                : launch_bwd_t<D, BF16, false, false>(p, maps, a, st);
}

cudaError_t launch_bwd(const sage_params &p, const __half *Q16, const __half *K16,
                       const void *V, const void *dO, const __half *dO16, BwdArgs a,
                       cudaStream_t st) {
    CUtensorMap maps[5];
    const uint64_t bh = static_cast<uint64_t>(p.B) * p.H;
    if (!make_tmap_3d(&maps[0], K16, p.d, p.N, bh) || !make_tmap_3d(&maps[1], V, p.d, p.N, bh) ||
        !make_tmap_3d(&maps[2], Q16, p.d, p.N, bh) || !make_tmap_3d(&maps[3], dO, p.d, p.N, bh) ||
        !make_tmap_3d(&maps[4], dO16, p.d, p.N, bh))
        return cudaErrorInvalidValue;
    const bool bf = p.dtype == SAGE_BF16;
    if (p.d == 128) return bf ? launch_bwd_d<128, true>(p, maps, a, st) : launch_bwd_d<128, false>(p, maps, a, st);
    return bf ? launch_bwd_d<64, true>(p, maps, a, st) : launch_bwd_d<64, false>(p, maps, a, st);
}

unsigned int take_bwd_error() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v));
    cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
    return v;
}

}  // namespace sage
