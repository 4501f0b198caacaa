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
//   S^T  = K^ Q^T    (M=128 keys, N=128 q, K=d)    TMEM R_S  = cols [0,128)
//   dP^T = V dO^T    (M=128 keys, N=128 q, K=d)    TMEM R_dP = cols [128,256)
//   dV_h = P^T_h dO^_h (A from TMEM, K=64 q)       TMEM R_V  = cols [256,384)  (h = q block)
//   dK_h = dS^T_h Q^_h (A from TMEM, K=64 q)       TMEM R_K  = cols [384,512)
//   dQ_g = dS^_g K^_g (A from smem, K=64 keys)     TMEM R_S (g = 0) / R_dP (g = 1), once their
//                                                  codes have been read by the dV / dK MMAs
// Warp roles (12 warps; registers 232 for the two math warpgroups, 40 for the control one):
//   warps 0-3  "score" warpgroup, thread = key: P = 2^(acc c - L2), dS = P o (dP - D) in place in
//              TMEM; per 64x64 tile max reductions; P and dS codes back into TMEM (A operands)
//              and dS codes into shared memory (A operand of dQ); dV rows in registers.
//   warps 4-7  "grad" warpgroup: dK rows in registers (thread = key); dQ products read with
//              thread = query row, scaled, and added to global dQ with vector float32 atomics.
//   warp 8     TMA producer; warp 9 TMEM allocation and the single MMA-issuing thread.
//
// Numerics (the CPU oracle mirrors these float32 steps):
//   c = fl32(fl32(sQ sK) * fl32(log2(e)/sqrt(d)));  L2 = fl32(L * fl32(log2(e)))
//   P = fl32(ex2(fl32(acc * c - L2)))   (with Q-smoothing ex2(fl32(fl32(acc * c + bias) - L2)))
//   dS = fl32(P * fl32(dP - D))
//   per 64x64 tile: s = fl32(max|x| / 127), code = rint(fl32(x * fl32(1/s))); max|x| < 2^-120 -> 0
#include "sage_device.cuh"
#include "sage_internal.h"

namespace sage {

__device__ unsigned int g_bwd_err;

namespace bwd {

constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kRegsMath = 232;
constexpr uint32_t kRegsControl = 40;
constexpr uint32_t R_S = 0, R_DP = 128, R_V = 256, R_K = 384;
constexpr float kTileZero = 7.52316384526264e-37f;   // 2^-120

template <int D>
struct Smem {
    alignas(1024) uint8_t kt[D / 64][128 * 128];    // K^ tile   [chunk of 64 d][key][128 B]
    alignas(1024) uint8_t vt[D / 64][128 * 128];    // V tile    (16-bit input type)
    alignas(1024) uint8_t qc[D / 64][128 * 128];    // Q^ chunk  [chunk][q row][128 B]
    alignas(1024) uint8_t doc[D / 64][128 * 128];   // dO chunk  (16-bit input type)
    alignas(1024) uint8_t dohc[D / 64][128 * 128];  // dO^ chunk (codes)
    alignas(1024) uint8_t dss[2][128 * 128];        // dS^ as MN-major A: [q block][key][64 q]
    float L2s[128], Ds[128];
    float red[4][2][4];                             // [warp][kb pair slot][4 maxima]
    float sds[2][2][2];                             // [chunk parity][kb][qb] dS tile scales
    float colsum[2][128];                           // [qb][key] column sums of dS (Q-smoothing)
    uint64_t kv_full, q_full, q_free, do_full, do_free, doh_full, doh_free;
    uint64_t s_full, dp_full, codes_ready, dss_free;
    uint64_t rv_full, rv_free, rk_full, rk_free, rs_full, rs_free, rdp_full, rdp_free;
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

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// code of x with reciprocal scale inv (inv = 0 for a zero tile)
__device__ __forceinline__ float tile_code(float x, float inv) {
    return fminf(127.0f, fmaxf(-127.0f, rintf(__fmul_rn(x, inv))));
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
                           &s.doh_free, &s.s_full, &s.dp_full, &s.dss_free, &s.rv_full, &s.rk_full,
                           &s.rs_full, &s.rdp_full, &s.mma_done};
        for (uint64_t *b : one) mbar_init(b, 1);
        mbar_init(&s.codes_ready, 4);
        mbar_init(&s.rv_free, 4);
        mbar_init(&s.rk_free, 4);
        mbar_init(&s.rs_free, 4);
        mbar_init(&s.rdp_free, 4);
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
                int nq = 0, ndo = 0, ndoh = 0;
                for (int it = 0; it < nmine; ++it) {
                    const int q0 = 128 * (c_first + it);
                    if (it > 0 && !mbar_wait(&s.do_free, (it - 1) & 1, abort_flag, &g_bwd_err, 1)) break;
                    mbar_arrive_expect_tx(&s.do_full, kTileBytes);
                    for (int c = 0; c < D / 64; ++c) tma_load_3d(s.doc[c], &mapdO, &s.do_full, 64 * c, q0, bh);
                    ndo = it + 1;
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
                if (nq > 0) mbar_wait_drain(&s.q_full, (nq - 1) & 1, &g_bwd_err, 4);
                if (ndoh > 0) mbar_wait_drain(&s.doh_full, (ndoh - 1) & 1, &g_bwd_err, 4);
            }
        } else if (warp == kMmaWarp) {
            // -------------------------------------------------------------- MMA issuer
            if (elect_one()) {
                constexpr uint32_t idKK = idesc_f16(128, 128, false, false, false);    // S^T
                constexpr uint32_t idDP = idesc_f16(128, 128, BF16, false, false);     // dP^T
                constexpr uint32_t idTS = idesc_f16(128, D, false, false, true);       // dV, dK
                constexpr uint32_t idQ = idesc_f16(128, D, false, true, true);         // dQ
                // base descriptors; a byte offset `off` inside an operand adds off >> 4
                const uint64_t dKt = sdesc_sw128(smem_u32(s.kt[0]), 16, 1024);
                const uint64_t dVt = sdesc_sw128(smem_u32(s.vt[0]), 16, 1024);
                const uint64_t dQc = sdesc_sw128(smem_u32(s.qc[0]), 16, 1024);
                const uint64_t dDo = sdesc_sw128(smem_u32(s.doc[0]), 16, 1024);
                const uint64_t dDoh = sdesc_sw128(smem_u32(s.dohc[0]), 16384, 1024);
                const uint64_t dQmn = sdesc_sw128(smem_u32(s.qc[0]), 16384, 1024);
                const uint64_t dKmn = sdesc_sw128(smem_u32(s.kt[0]), 16384, 1024);
                const uint64_t dDss = sdesc_sw128(smem_u32(s.dss[0]), 16384, 1024);
                bool ok = mbar_wait(&s.kv_full, 0, abort_flag, &g_bwd_err, 5);
                for (int it = 0; it < nmine && ok; ++it) {
                    const uint32_t ph = it & 1;
                    // S^T = K^ Q^T
                    if (!mbar_wait(&s.q_full, ph, abort_flag, &g_bwd_err, 6)) break;
                    if (it > 0 && !mbar_wait(&s.rs_free, (it - 1) & 1, abort_flag, &g_bwd_err, 7)) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        umma_ss(tmem + R_S, dKt + o, dQc + o, idKK, kk > 0);
                    }
                    umma_commit(&s.s_full);
                    // dP^T = V dO^T
                    if (!mbar_wait(&s.do_full, ph, abort_flag, &g_bwd_err, 8)) break;
                    if (it > 0 && !mbar_wait(&s.rdp_free, (it - 1) & 1, abort_flag, &g_bwd_err, 9)) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        umma_ss(tmem + R_DP, dVt + o, dDo + o, idDP, kk > 0);
                    }
                    umma_commit(&s.dp_full);
                    umma_commit(&s.do_free);
                    // the score warpgroup turns S^T, dP^T into P / dS codes
                    if (!mbar_wait(&s.codes_ready, ph, abort_flag, &g_bwd_err, 10)) break;
                    if (!mbar_wait(&s.doh_full, ph, abort_flag, &g_bwd_err, 11)) break;
                    tc_fence_after();
                    for (int h = 0; h < 2 && ok; ++h) {
                        // dV_h = P^T[:, h] dO^_h  -> R_V
                        const int uv = 2 * it + h;
                        if (uv > 0 && !mbar_wait(&s.rv_free, (uv - 1) & 1, abort_flag, &g_bwd_err, 12)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ts(tmem + R_V, tmem + R_S + 32 * h + 8 * kk, dDoh + (((64 * h + 16 * kk) * 128) >> 4), idTS, kk > 0);
                        umma_commit(&s.rv_full);
                        // dK_h = dS^T[:, h] Q^_h  -> R_K
                        if (uv > 0 && !mbar_wait(&s.rk_free, (uv - 1) & 1, abort_flag, &g_bwd_err, 13)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ts(tmem + R_K, tmem + R_DP + 32 * h + 8 * kk, dQmn + (((64 * h + 16 * kk) * 128) >> 4), idTS, kk > 0);
                        umma_commit(&s.rk_full);
                    }
                    if (!ok) break;
                    umma_commit(&s.doh_free);
                    umma_commit(&s.q_free);
                    // dQ_g = dS^[:, keys of g] K^_g -> R_S (g = 0), R_DP (g = 1); the tensor pipe
                    // runs in issue order, so the codes these regions held are already consumed
#pragma unroll 1
                    for (int g = 0; g < 2; ++g) {
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t o = ((64 * g + 16 * kk) * 128) >> 4;
                            umma_ss(tmem + (g ? R_DP : R_S), dDss + o, dKmn + o, idQ, kk > 0);
                        }
                        umma_commit(g ? &s.rdp_full : &s.rs_full);
                    }
                    umma_commit(&s.dss_free);
                }
                umma_commit(&s.mma_done);
                mbar_wait_drain(&s.mma_done, 0, &g_bwd_err, 14);
            }
        }
    } else if (warp < 4) {
        regs_inc<kRegsMath>();
        // ------------------------------------------------------------------ score warpgroup
        const int tq = threadIdx.x;                       // 0..127: key lane / query index
        const int quarter = warp;
        const int key = k0 + tq;                          // key index within the head
        const int kb = tq >> 6;                           // key block of this lane (0/1)
        const int kblk = min(key, N - 1) >> 6;            // global key block
        const bool key_ok = key < N;
        const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
        const float sk = a.sK[static_cast<size_t>(bh) * nblk + kblk];
        float dv[D];
#pragma unroll
        for (int c = 0; c < D; ++c) dv[c] = 0.0f;
        for (int it = 0; it < nmine; ++it) {
            const uint32_t ph = it & 1;
            const int ic = c_first + it;
            const int q0 = 128 * ic;
            // per-chunk row data: L2 = fl32(L log2 e), D
            {
                const int r = q0 + tq;
                s.L2s[tq] = r < N ? __fmul_rn(a.L[bhN + r], kLog2e) : 0.0f;
                s.Ds[tq] = r < N ? a.D[bhN + r] : 0.0f;
            }
            named_bar_sync(1, 128);
            float cq[2], biasv[2] = {0.0f, 0.0f};
            int qblk[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                qblk[h] = min(2 * ic + h, nblk - 1);
                cq[h] = __fmul_rn(__fmul_rn(a.sQ[static_cast<size_t>(bh) * nblk + qblk[h]], sk), a.sl2);
                if (BIAS && key_ok) biasv[h] = a.qbias[(static_cast<size_t>(bh) * nblk + qblk[h]) * N + key];
            }
            // valid query columns for this key: [qlo, qhi) relative to q0
            const int qhi = min(128, N - q0);
            const int qlo = a.causal ? max(0, key - q0) : 0;
            if (!mbar_wait(&s.s_full, ph, abort_flag, &g_bwd_err, 20)) break;
            if (!mbar_wait(&s.dp_full, ph, abort_flag, &g_bwd_err, 21)) break;
            tc_fence_after();
            // pass 1: P and dS in place, tile maxima, column sums of dS
            float mp[2] = {0.0f, 0.0f}, md[2] = {0.0f, 0.0f}, cs[2] = {0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll 1
            for (int cc = 64 * h; cc < 64 * h + 64; cc += 16) {
                uint32_t sr[16], dr[16];
                tmem_ld16(lane_base + R_S + cc, sr);
                tmem_ld16(lane_base + R_DP + cc, dr);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int col = cc + k;
                    const float acc = __uint_as_float(sr[k]);
                    float x;
                    if (BIAS) x = __fsub_rn(__fmaf_rn(acc, cq[h], biasv[h]), s.L2s[col]);
                    else x = __fmaf_rn(acc, cq[h], -s.L2s[col]);
                    const bool ok = key_ok && col >= qlo && col < qhi;
                    const float p = ok ? ex2_approx(x) : 0.0f;
                    const float ds = __fmul_rn(p, __fsub_rn(__uint_as_float(dr[k]), s.Ds[col]));
                    mp[h] = fmaxf(mp[h], p);
                    md[h] = fmaxf(md[h], fabsf(ds));
                    cs[h] += ds;
                    if (DUMP) {
                        if (ok) a.dump_s[(bhN + q0 + col) * N + key] = static_cast<int32_t>(acc);
                    }
                    sr[k] = __float_as_uint(p);
                    dr[k] = __float_as_uint(ds);
                }
                tmem_st16(lane_base + R_S + cc, sr);
                tmem_st16(lane_base + R_DP + cc, dr);
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
                s.red[warp][it & 1][0] = mp[0];
                s.red[warp][it & 1][1] = mp[1];
                s.red[warp][it & 1][2] = md[0];
                s.red[warp][it & 1][3] = md[1];
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
                const float mxp = fmaxf(s.red[w0][it & 1][h], s.red[w0 + 1][it & 1][h]);
                const float mxd = fmaxf(s.red[w0][it & 1][2 + h], s.red[w0 + 1][it & 1][2 + h]);
                sp[h] = mxp < kTileZero ? 0.0f : __fdiv_rn(mxp, 127.0f);
                ip[h] = mxp < kTileZero ? 0.0f : __frcp_rn(sp[h]);
                sd[h] = mxd < kTileZero ? 0.0f : __fdiv_rn(mxd, 127.0f);
                id[h] = mxd < kTileZero ? 0.0f : __frcp_rn(sd[h]);
            }
            if ((tq & 63) == 0) {
                s.sds[it & 1][kb][0] = sd[0];
                s.sds[it & 1][kb][1] = sd[1];
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
                    const float p0 = tile_code(__uint_as_float(pr[k]), ip[h]);
                    const float p1 = tile_code(__uint_as_float(pr[k + 1]), ip[h]);
                    const float d0 = tile_code(__uint_as_float(dr[k]), id[h]);
                    const float d1 = tile_code(__uint_as_float(dr[k + 1]), id[h]);
                    pk[k / 2] = pack_half2(p0, p1);
                    dk[k / 2] = pack_half2(d0, d1);
                    if (DUMP) {
                        const int col = cc + k;
                        if (key_ok && q0 + col < N) {
                            a.dump_p[(bhN + q0 + col) * N + key] = static_cast<int16_t>(p0);
                            a.dump_ds[(bhN + q0 + col) * N + key] = static_cast<int16_t>(d0);
                        }
                        if (key_ok && q0 + col + 1 < N) {
                            a.dump_p[(bhN + q0 + col + 1) * N + key] = static_cast<int16_t>(p1);
                            a.dump_ds[(bhN + q0 + col + 1) * N + key] = static_cast<int16_t>(d1);
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
            // dV += s_P s_dO (P^T dO^)_h
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int uv = 2 * it + h;
                if (!mbar_wait(&s.rv_full, uv & 1, abort_flag, &g_bwd_err, 23)) break;
                tc_fence_after();
                const float sc = __fmul_rn(sp[h], a.sdO[static_cast<size_t>(bh) * nblk + qblk[h]]);
#pragma unroll
                for (int cc = 0; cc < D; cc += 16) {
                    uint32_t r[16];
                    tmem_ld16(lane_base + R_V + cc, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) dv[cc + k] = __fmaf_rn(sc, __uint_as_float(r[k]), dv[cc + k]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(&s.rv_free);
            }
        }
        if (key_ok && !*abort_flag) {
            float *dst = a.dV + (bhN + key) * D;
#pragma unroll
            for (int c = 0; c < D; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(dv[c], dv[c + 1], dv[c + 2], dv[c + 3]);
        }
    } else {
        regs_inc<kRegsMath>();
        // ------------------------------------------------------------------ grad warpgroup
        const int tq = threadIdx.x - 128;                 // key lane (dK) / query lane (dQ)
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
        for (int g = 0; g < 2; ++g) skb[g] = a.sK[static_cast<size_t>(bh) * nblk + min(2 * jt + g, nblk - 1)];
        for (int it = 0; it < nmine; ++it) {
            const int ic = c_first + it;
            const int q0 = 128 * ic;
            int qblk[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) qblk[h] = min(2 * ic + h, nblk - 1);
            // dK += s_dS s_Q / sqrt(d) (dS^T Q^)_h   (+ Q-smoothing bias (dS^T 1) mu_Q / sqrt(d))
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int uk = 2 * it + h;
                if (!mbar_wait(&s.rk_full, uk & 1, abort_flag, &g_bwd_err, 30)) break;
                tc_fence_after();
                const float sc = __fmul_rn(__fmul_rn(s.sds[it & 1][kb][h], a.sQ[static_cast<size_t>(bh) * nblk + qblk[h]]), a.inv_sqrt_d);
#pragma unroll
                for (int cc = 0; cc < D; cc += 16) {
                    uint32_t r[16];
                    tmem_ld16(lane_base + R_K + cc, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) dk[cc + k] = __fmaf_rn(sc, __uint_as_float(r[k]), dk[cc + k]);
                }
                if (BIAS && q0 + 64 * h < N) {
                    const float w = __fmul_rn(s.colsum[h][tq], a.inv_sqrt_d);
                    const float *mu = a.muQ + (static_cast<size_t>(bh) * nblk + qblk[h]) * D;
#pragma unroll
                    for (int c = 0; c < D; ++c) dk[c] = __fmaf_rn(w, mu[c], dk[c]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(&s.rk_free);
            }
            // dQ rows: thread = query row of the chunk
            const int qrow = q0 + tq;
            const int h_row = tq >> 6;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint64_t *full = g ? &s.rdp_full : &s.rs_full;
                uint64_t *freeb = g ? &s.rdp_free : &s.rs_free;
                if (!mbar_wait(full, it & 1, abort_flag, &g_bwd_err, 31)) break;
                tc_fence_after();
                const float sc = __fmul_rn(__fmul_rn(s.sds[it & 1][g][h_row], skb[g]), a.inv_sqrt_d);
                const bool live = qrow < N && k0 + 64 * g < N;
                float *dst = a.dQ + (bhN + min(qrow, N - 1)) * D;
#pragma unroll
                for (int cc = 0; cc < D; cc += 16) {
                    uint32_t r[16];
                    tmem_ld16(lane_base + (g ? R_DP : R_S) + cc, r);
                    tmem_wait_ld();
                    if (live) {
#pragma unroll
                        for (int k = 0; k < 16; k += 4)
                            red_add_v4(dst + cc + k, sc * __uint_as_float(r[k]), sc * __uint_as_float(r[k + 1]),
                                       sc * __uint_as_float(r[k + 2]), sc * __uint_as_float(r[k + 3]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane_id() == 0) mbar_arrive(freeb);
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
