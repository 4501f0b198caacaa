// sage_quant.cu -- smoothing, per-block INT8 quantisation and the streaming helper passes.
//
// "SageBwd: A Trainable Low-bit Attention" (structured summary): prerequisites, INT8 quantisation
// (X^ = round(X / delta), delta = max|X| / 127, per-block granularity aligned with the attention
// tiles) and K-/Q-smoothing (mu_K = mean over tokens of K, K_sm = K - mu_K; mu_Qi = mean over the
// rows of query block i); method steps, forward (2) and backward (1).
// "SageAttention3 ..." (review), eq. (7).
//
// Bit-exact contract:
//   block        = 64 tokens x d
//   mu           = float64 sum, float64 divide, one rounding to float32
//   x            = fl32(v - mu)
//   delta        = fl32(max|x| / 127)        (IEEE division, __fdiv_rn)
//   code         = clamp(rint_half_even(fl32(x / delta)), -127, 127), zero block -> delta 0, code 0
// FP8 variant ("SageAttention3 ..." (review), INT8 vs FP8 training): delta = fl32(max|x| / 448)
// and code = E4M3(fl32(x / delta)), round to nearest even, saturating at +-448.
// QK-norm prologue ("SageBwd ..." (structured summary), QK-norm; norm epsilon 1e-6): Q and K rows
// become y = rnd16(fl32(fl32(x r) gamma_c)), r the float32 nearest to 1 / sqrt(S / d + eps) with
// S the exact sum of x^2, before the K-mean, the smoothing and the quantiser see them.
//
// All kernels here stream through HBM once; they are bound by memory bandwidth.
#include "sage_device.cuh"
#include "sage_internal.h"

namespace sage {

// ---------------------------------------------------------------------------------------------
// element loads: 8 consecutive 16-bit values -> 8 floats (exact)
// ---------------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 f = __half22float2(h);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        } else {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            float2 f = __bfloat1622float2(h);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

// 8 consecutive 16-bit values (one 16-byte word) -> 8 floats (exact)
template <typename T>
__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<T, __half>::value) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        } else {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

__device__ __forceinline__ int quant_code(float x, float delta) {
    if (delta == 0.0f) return 0;
    int q = __float2int_rn(__fdiv_rn(x, delta));
    return q > 127 ? 127 : (q < -127 ? -127 : q);
}

__device__ __forceinline__ uint2 pack_codes8(const float (&x)[8], float delta) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= (static_cast<uint32_t>(quant_code(x[i], delta)) & 0xFFu) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= (static_cast<uint32_t>(quant_code(x[4 + i], delta)) & 0xFFu) << (8 * i);
    return make_uint2(lo, hi);
}

// E4M3 codes of 8 values (bit patterns, 8 bytes); delta = 0 gives all-zero codes
__device__ __forceinline__ uint2 pack_codes8_e4m3(const float (&x)[8], float delta) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = delta == 0.0f ? 0u : e4m3x2(__fdiv_rn(x[2 * i], delta), __fdiv_rn(x[2 * i + 1], delta));
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// E4M3 codes of 8 values and, in *h16, their fp16 values: one division a value, the fp16 value
// converted from the code (every E4M3 value is exact in fp16)
__device__ __forceinline__ uint2 pack_codes8_e4m3_h16(const float (&x)[8], float delta, uint4 *h16) {
    uint32_t w[4], h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint16_t c = delta == 0.0f ? static_cast<uint16_t>(0)
                                         : e4m3x2(__fdiv_rn(x[2 * i], delta), __fdiv_rn(x[2 * i + 1], delta));
        w[i] = c;
        h[i] = e4m3x2_to_f16x2(c);
    }
    *h16 = make_uint4(h[0], h[1], h[2], h[3]);
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// integer-valued fp16 copies of the codes (the tensor-core operand format on sm_103a)
__device__ __forceinline__ uint4 pack_codes8_f16(const float (&x)[8], float delta) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __halves2half2(__int2half_rn(quant_code(x[2 * i], delta)),
                                   __int2half_rn(quant_code(x[2 * i + 1], delta)));
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__device__ __forceinline__ float round_to(float y);
template <>
__device__ __forceinline__ float round_to<__half>(float y) { return __half2float(__float2half_rn(y)); }
template <>
__device__ __forceinline__ float round_to<__nv_bfloat16>(float y) { return __bfloat162float(__float2bfloat16_rn(y)); }

// s + e = a + b exactly (Knuth's two-sum; the error term does not depend on the operand order)
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// A sum of float32 values kept as an unevaluated triple h + l + t: two-sums make every step exact
// but the additions into t (relative 2^-65 over thousands of terms).  bf16 inputs are exact in
// float32, so this replaces per-element float64 additions (slow on GB300) at no loss of accuracy;
// the sum must stay below the float32 range.
struct Sum3 {
    float h = 0.0f, l = 0.0f, t = 0.0f;
    __device__ __forceinline__ void add(float v) {
        float e1, e2;
        two_sum(h, v, h, e1);
        two_sum(l, e1, l, e2);
        t = __fadd_rn(t, e2);
    }
    __device__ __forceinline__ double value() const {
        return (static_cast<double>(h) + static_cast<double>(l)) + static_cast<double>(t);
    }
};

// r = the float32 nearest to 1 / sqrt(v), v = S / d + eps, with S = h + l + t the exact sum of
// squares held as an unevaluated float32 triple and d a power of two.
//   1. v as a float32 pair vh + vl (two-sums; relative error about 2^-46) and a candidate
//      r0 = fl32(1 / fl32(sqrt(vh))), within about two ulps of the exact value r*.
//   2. The residual rho = 1 - r0^2 v in compensated float32: r0^2 = a + b exactly (a two-product
//      by fused multiply-add), then 1 - a vh, - b vh and - a vl by fused multiply-adds; |rho| is
//      below about 2^-21 and its error below about 2^-43.
//   3. r* = r0 (1 - rho)^(-1/2) = r0 (1 + rho/2 + 3 rho^2 / 8 + O(rho^3)), so r* lies
//      z = (rho/2 + 3 rho^2/8) r0 / ulp(r0) ulps above r0, z known to within about 2^-19.
//      The nearest float32 is r0 + rint(z) ulp.
//   4. Where z lies within 2^-16 of a half-integer (about one row in 10 000), or in the corner
//      cases (|rint(z)| > 2, r0 within four ulps of either end of its binade, v outside
//      [2^-100, 2^100]), float64 decides:
//      fl32(1 / sqrt(fl64(S / d + eps))) with the IEEE float64 square root and division.
__device__ __noinline__ float rsqrt_rn_fallback(float h, float l, float t, int d, float eps) {
    const double S = (static_cast<double>(h) + static_cast<double>(l)) + static_cast<double>(t);
    const double v = fma(S, 1.0 / static_cast<double>(d), static_cast<double>(eps));
    return static_cast<float>(1.0 / sqrt(v));
}

__device__ __forceinline__ float rsqrt_rn(float h, float l, float t, int d, float eps) {
    const float inv_d = 1.0f / static_cast<float>(d);              // exact: d = 64 or 128
    float s1, e1, sh, sl;
    two_sum(h, l, s1, e1);
    two_sum(s1, __fadd_rn(e1, t), sh, sl);                         // S = sh + sl
    sh = __fmul_rn(sh, inv_d);
    sl = __fmul_rn(sl, inv_d);
    float a1, b1, vh, vl;
    two_sum(sh, eps, a1, b1);
    two_sum(a1, __fadd_rn(b1, sl), vh, vl);                        // v = vh + vl
    if (!(vh >= 0x1p-100f && vh <= 0x1p100f)) return rsqrt_rn_fallback(h, l, t, d, eps);
    const float r0 = __frcp_rn(__fsqrt_rn(vh));
    const float a = __fmul_rn(r0, r0);
    const float b = __fmaf_rn(r0, r0, -a);                         // r0^2 = a + b
    float rho = __fmaf_rn(-a, vh, 1.0f);
    rho = __fmaf_rn(-b, vh, rho);
    rho = __fmaf_rn(-a, vl, rho);
    const float rel = __fmaf_rn(__fmul_rn(0.375f, rho), rho, __fmul_rn(0.5f, rho));
    const uint32_t mant = __float_as_uint(r0) & 0x7FFFFFu;
    const float z = __fmul_rn(rel, static_cast<float>(mant | 0x800000u));   // r0 / ulp(r0) = 1.mant * 2^23
    const float k = rintf(z);
    // candidates and midpoints up to 2.5 ulps away keep r0's spacing when r0 is at least four
    // ulps from both ends of its binade
    if (fabsf(__fsub_rn(fabsf(__fsub_rn(z, k)), 0.5f)) < 0x1p-16f || fabsf(k) > 2.0f || mant < 4u ||
        mant > 0x7FFFFBu)
        return rsqrt_rn_fallback(h, l, t, d, eps);
    const float ulp = __uint_as_float(__float_as_uint(r0) & 0x7F800000u) * 0x1p-23f;
    return __fmaf_rn(k, ulp, r0);                                  // exact: r0 or a neighbour
}

// QK-norm of this lane's 8 values of a row whose d / 8 slices sit in `lanes` consecutive lanes
// (every lane of the warp takes part).  The squares of 16-bit values are exact in float32 (bf16:
// for 2^-63 <= |x| < 2^63).  They are summed as an unevaluated float32 triple h + l + t with
// two-sums, whose only rounding is in t (relative 2^-65 over a row); a butterfly of the same
// exact steps leaves the same triple in every lane of the row.
// Returns r, the float32 nearest to 1 / sqrt(S / d + eps) (rsqrt_rn), and replaces v by
// rnd_T(fl32(fl32(v r) g_c)).
template <typename T>
__device__ __forceinline__ float qk_norm8(float (&v)[8], const float *gamma, int c0, int lanes,
                                          int d, float eps) {
    float h = 0.0f, l = 0.0f, t = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float e1, e2;
        two_sum(h, __fmul_rn(v[i], v[i]), h, e1);
        two_sum(l, e1, l, e2);
        t = __fadd_rn(t, e2);
    }
    for (int o = 1; o < lanes; o <<= 1) {
        const float ho = __shfl_xor_sync(0xffffffffu, h, o);
        const float lo = __shfl_xor_sync(0xffffffffu, l, o);
        const float to = __shfl_xor_sync(0xffffffffu, t, o);
        float e1, e2, e3;
        two_sum(h, ho, h, e1);
        two_sum(l, lo, l, e2);
        two_sum(l, e1, l, e3);
        t = __fadd_rn(__fadd_rn(__fadd_rn(t, to), e2), e3);
    }
    const float r = rsqrt_rn(h, l, t, d, eps);
    float g[8] = {1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f};
    if (gamma) {
        *reinterpret_cast<float4 *>(&g[0]) = *reinterpret_cast<const float4 *>(gamma + c0);
        *reinterpret_cast<float4 *>(&g[4]) = *reinterpret_cast<const float4 *>(gamma + c0 + 4);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float y = __fmul_rn(v[i], r);
        if (gamma) y = __fmul_rn(y, g[i]);
        v[i] = round_to<T>(y);
    }
    return r;
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]);
template <>
__device__ __forceinline__ uint4 pack8<__half>(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ uint4 pack8<__nv_bfloat16>(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Block-wide max of non-negative floats (256 threads).
__device__ __forceinline__ float block_max_256(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    return m;
}

// 16-byte read-only global load; volatile so that a batch of them is issued in program order,
// all before the first use
__device__ __forceinline__ uint4 ldg128_nc(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// fp16 value as an exact integer multiple of 2^-24 (the smallest fp16 subnormal): every finite
// fp16 is m 2^-24 (subnormal) or (1024 + m) 2^(e - 25), so the multiple is m or
// (1024 + m) << (e - 1), below 2^40 in magnitude.
__device__ __forceinline__ long long half_fixed24(uint32_t h) {
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    const long long mag = e == 0 ? static_cast<long long>(m) : static_cast<long long>(1024u | m) << (e - 1);
    return (h & 0x8000u) ? -mag : mag;
}

// ---------------------------------------------------------------------------------------------
// a1 (FP4 quantiser): partial sums of K over token ranges, exact, one (head, split) per CTA.
// partial[(bh * S + s) * d + c] = sum_{n in split s} K[bh, n, c]
// fp16 input: int64 multiples of 2^-24 (integer adds, far faster than float64 ones here and just
// as exact: a sum of 32768 values stays below 2^55, and any sum below 2^53 is exact in both);
// bf16 input (exponent range of float32): float32 two-sum triples per thread, turned into float64
// once (see Sum3).  Both occupy 8 bytes per entry.
// ---------------------------------------------------------------------------------------------
// With QK-norm (NORM) the rows are normalised first; the loop then runs warp-uniform trip counts
// (rows past the split are zeros and not added) because the norm's shuffles need every lane.
template <typename T, bool NORM>
__global__ void __launch_bounds__(256) kmean_partial_kernel(const T *__restrict__ K,
                                                            double *__restrict__ partial, int N,
                                                            int d, int S, int rows_per_split,
                                                            const float *__restrict__ gamma, float eps) {
    if constexpr (NORM) {
        __shared__ double redn[256 * 8];
        const int bh = blockIdx.x, s = blockIdx.y;
        const int vec_per_row = d / 8;
        const int rows_in_flight = 256 / vec_per_row;
        const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
        const int n0 = s * rows_per_split;
        const int n1 = min(N, n0 + rows_per_split);
        long long acci[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        Sum3 accd[8];
        const T *base = K + static_cast<size_t>(bh) * N * d;
        // unrolled: the norm's two-sum chains of several rows overlap
#pragma unroll 4
        for (int b0 = n0; b0 < n1; b0 += rows_in_flight) {
            const int n = b0 + rg;
            float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (n < n1) load8(base + static_cast<size_t>(n) * d + cv * 8, v);
            qk_norm8<T>(v, gamma, cv * 8, vec_per_row, d, eps);
            if (n < n1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if constexpr (std::is_same<T, __half>::value)
                        acci[i] += half_fixed24(__half_as_ushort(__float2half_rn(v[i])));
                    else
                        accd[i].add(v[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if constexpr (std::is_same<T, __half>::value)
                reinterpret_cast<long long *>(redn)[threadIdx.x * 8 + i] = acci[i];
            else
                redn[threadIdx.x * 8 + i] = accd[i].value();
        }
        __syncthreads();
        if (threadIdx.x < d) {
            const int c = threadIdx.x, cvv = c / 8, ci = c % 8;
            if constexpr (std::is_same<T, __half>::value) {
                long long sum = 0;
                for (int g = 0; g < rows_in_flight; ++g) sum += reinterpret_cast<long long *>(redn)[(g * vec_per_row + cvv) * 8 + ci];
                reinterpret_cast<long long *>(partial)[(static_cast<size_t>(bh) * S + s) * d + c] = sum;
            } else {
                double sum = 0.0;
                for (int g = 0; g < rows_in_flight; ++g) sum += redn[(g * vec_per_row + cvv) * 8 + ci];
                partial[(static_cast<size_t>(bh) * S + s) * d + c] = sum;
            }
        }
    } else if constexpr (std::is_same<T, __half>::value) {
        // fp16 values v = hi + lo exactly, hi = v rounded to a multiple of 2^-4 (adding 1.5 2^19
        // rounds there) and lo = v - hi, a multiple of 2^-24 with |lo| <= 2^-5.  Sixteen his stay
        // below 2^20 (multiples of 2^-4: 24 bits) and sixteen los below 2^-1 (multiples of
        // 2^-24: 23 bits), so packed float32 adds sum them exactly; every sixteen rows both join
        // the int64 total in units of 2^-24.
        __shared__ long long redi[256 * 8];
        const int bh = blockIdx.x, s = blockIdx.y;
        const int vec_per_row = d / 8;
        const int rows_in_flight = 256 / vec_per_row;
        const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
        const int n0 = s * rows_per_split;
        const int n1 = min(N, n0 + rows_per_split);
        long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        const T *base = K + static_cast<size_t>(bh) * N * d + cv * 8;
        const f2 c2{786432.0f, 786432.0f};               // 1.5 * 2^19
        for (int nb = n0 + rg; nb < n1; nb += 16 * rows_in_flight) {
            f2 hs[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
            f2 ls[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
            // all sixteen rows' loads in flight before any is used (rows past the split are zeros)
            uint4 w[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int n = nb + u * rows_in_flight;
                w[u] = n < n1 ? ldg128_nc(base + static_cast<size_t>(n) * d) : make_uint4(0, 0, 0, 0);
            }
            // (every use below depends on this statement, which comes after the last load)
#pragma unroll
            for (int u = 0; u < 16; ++u) asm volatile("" : "+r"(w[u].x), "+r"(w[u].y), "+r"(w[u].z), "+r"(w[u].w));
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                float v[8];
                unpack8<T>(w[u], v);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const f2 x{v[2 * i], v[2 * i + 1]};
                    const f2 hi = sub2(add2(x, c2), c2);
                    hs[i] = add2(hs[i], hi);
                    ls[i] = add2(ls[i], sub2(x, hi));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += (__float2ll_rn(hs[i].x * 16.0f) << 20) + __float2ll_rn(ls[i].x * 16777216.0f);
                acc[2 * i + 1] += (__float2ll_rn(hs[i].y * 16.0f) << 20) + __float2ll_rn(ls[i].y * 16777216.0f);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) redi[threadIdx.x * 8 + i] = acc[i];
        __syncthreads();
        if (threadIdx.x < d) {
            const int c = threadIdx.x, cvv = c / 8, ci = c % 8;
            long long sum = 0;
            for (int g = 0; g < rows_in_flight; ++g) sum += redi[(g * vec_per_row + cvv) * 8 + ci];
            reinterpret_cast<long long *>(partial)[(static_cast<size_t>(bh) * S + s) * d + c] = sum;
        }
    } else {
        __shared__ double red[256 * 8];
        const int bh = blockIdx.x, s = blockIdx.y;
        const int vec_per_row = d / 8;                    // threads per row
        const int rows_in_flight = 256 / vec_per_row;
        const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
        const int n0 = s * rows_per_split;
        const int n1 = min(N, n0 + rows_per_split);
        Sum3 acc[8];
        const T *base = K + static_cast<size_t>(bh) * N * d;
        // unrolled so that several rows' loads are in flight at once
#pragma unroll 4
        for (int n = n0 + rg; n < n1; n += rows_in_flight) {
            float v[8];
            load8(base + static_cast<size_t>(n) * d + cv * 8, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i].add(v[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) red[threadIdx.x * 8 + i] = acc[i].value();
        __syncthreads();
        if (threadIdx.x < d) {
            const int c = threadIdx.x, cvv = c / 8, ci = c % 8;
            double sum = 0.0;
            for (int g = 0; g < rows_in_flight; ++g) sum += red[(g * vec_per_row + cvv) * 8 + ci];
            partial[(static_cast<size_t>(bh) * S + s) * d + c] = sum;
        }
    }
}

// (FP4 quantiser) Per-channel mean that tensor z of 64-row block blk has subtracted before quantisation, into
// mu_s: mu_K from the K-mean partial sums (z = 1 with smooth_k), or the block's own mean of Q
// (z = 0 with smooth_q; with NORM the rows pass through the QK-norm first).  Writes muK / muQ and
// returns whether the tensor is smoothed.  Ends with a CTA barrier.
// The fields of the kernel parameter the helper reads, by value (a reference to the parameter
// itself would copy it to local memory).
struct SmoothIn {
    const double *kpartial;
    float *muK, *muQ;
    int ksplits, N, d, smooth_k, smooth_q;
};

template <typename T, bool NORM>
__device__ __forceinline__ bool smoothing_mean(const SmoothIn a, const T *src, int z, int blk,
                                               int bh, size_t blk_off, int cv, int rg,
                                               int vec_per_row, int rows_in_flight, int iters,
                                               const float *gamma, float eps, float *mu_s,
                                               double *colsum) {
    const int d = a.d, N = a.N;
    const bool norm = NORM && z < 2;
    // per-channel mean to subtract (zero when this tensor is not smoothed)
    bool smooth = false;
    if (z == 1 && a.smooth_k) {
        smooth = true;
        if (threadIdx.x < d) {
            const double *p = a.kpartial + static_cast<size_t>(bh) * a.ksplits * d + threadIdx.x;
            double sum = 0.0;
            if constexpr (std::is_same<T, __half>::value) {
                // exact int64 multiples of 2^-24 (see kmean_partial_kernel)
                long long si = 0;
                for (int s = 0; s < a.ksplits; ++s) si += reinterpret_cast<const long long *>(p)[static_cast<size_t>(s) * d];
                sum = static_cast<double>(si) * 0x1p-24;
            } else {
                for (int s = 0; s < a.ksplits; ++s) sum += p[static_cast<size_t>(s) * d];
            }
            const float mu = static_cast<float>(sum / static_cast<double>(N));
            mu_s[threadIdx.x] = mu;
            if (blk == 0 && a.muK) a.muK[static_cast<size_t>(bh) * d + threadIdx.x] = mu;
        }
    } else if (z == 0 && a.smooth_q) {
        smooth = true;
        // per thread: fp16 values as exact int64 multiples of 2^-24 (no float64 adds, slow on
        // GB300); bf16 in float64 (a float32 triple here would cost the plain kernel registers)
        long long acci[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        double accd[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int it = 0; it < iters; ++it) {
            const int r = rg + it * rows_in_flight;
            float v[8];
            load8(src + blk_off + static_cast<size_t>(r) * d + cv * 8, v);
            if (norm) qk_norm8<T>(v, gamma, cv * 8, vec_per_row, d, eps);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if constexpr (std::is_same<T, __half>::value)
                    acci[i] += half_fixed24(__half_as_ushort(__float2half_rn(v[i])));
                else
                    accd[i] += static_cast<double>(v[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if constexpr (std::is_same<T, __half>::value)
                colsum[threadIdx.x * 8 + i] = static_cast<double>(acci[i]) * 0x1p-24;
            else
                colsum[threadIdx.x * 8 + i] = accd[i];
        }
        __syncthreads();
        if (threadIdx.x < d) {
            const int c = threadIdx.x, cvv = c / 8, ci = c % 8;
            double sum = 0.0;
            for (int g = 0; g < rows_in_flight; ++g) sum += colsum[(g * vec_per_row + cvv) * 8 + ci];
            const float mu = static_cast<float>(sum / 64.0);
            mu_s[c] = mu;
            a.muQ[(static_cast<size_t>(bh) * (N / 64) + blk) * d + c] = mu;
        }
    } else if (z == 1 && a.muK && blk == 0 && threadIdx.x < d) {
        a.muK[static_cast<size_t>(bh) * d + threadIdx.x] = 0.0f;
    }
    __syncthreads();

    return smooth;
}

// ---------------------------------------------------------------------------------------------
// a1 + a2: the K-mean, the smoothing and the per-block quantisation of Q (z=0), K (z=1), V (z=2)
// in one persistent, pipelined pass.
//
// Every 64 x d block is contiguous in memory, so one bulk copy (cp.async.bulk, completion counted
// in bytes on an mbarrier) brings it into a shared-memory stage; the stages keep the next blocks'
// loads in flight while the CTA works on the current one.  A CTA walks one sequence of blocks:
//   1. (K-smoothing) its contiguous share of K's blocks, summed column by column into one partial
//      sum per head it touches (exact: int64 multiples of 2^-24 for fp16; float32 triples, then
//      float64, for bf16), stored at slot (CTA + head), which no other CTA uses.  The last CTA to
//      add a partial of head h adds all of them in CTA order, writes mu_K = fl32(sum / N) and
//      raises the head's flag;
//   2. the blocks w = blockIdx.x + j gridDim.x of K, Q, V in that order (K's blocks first: the
//      K-mean has just read them and most are still in L2), each smoothed, reduced to its
//      maximum |x| and written as codes; a K block first waits for its head's flag (a
//      cooperative launch keeps every CTA resident, so every flag is raised).
//
// Codes: rne(fl32(x / delta)) is taken as q = fl32(x r), r = fl32(1 / delta), rounded to the
// nearest integer k.  For normal delta, |q - x/delta| < 2^-16 and |fl32(x/delta) - x/delta| <=
// 2^-18 (|x/delta| <= 127 / (1 - 2^-24)), so where q lies more than 2^-15 from a half-integer
// (|q - k| < 1/2 - 2^-15) both x / delta and its rounding lie on k's side of it and k is the code.
// Eight values whose q comes nearer (about 6e-5 of them), or a subnormal delta, take the
// correctly rounded division itself.
// ---------------------------------------------------------------------------------------------
constexpr int kQuantThreads = 256;
// CTAs per SM (the QK-norm variants, which need more registers, keep two).  Measured with the L2
// flushed between calls: two 0.0959 ms, three 0.0928, four 0.0980 at B2 H16 N8192 d128; two
// 0.1338, three 0.1154 at B2 H32 N8192 d64.
constexpr int kQuantCtas = 3;
// bytes of block stages per CTA: 3 x 16 KB at d = 128
constexpr int kQuantStageBytes = 49152;
constexpr int kQuantMaxStages = 8;
constexpr int kQuantGridMax = kQuantCtas * 152;   // CTAs of the pass at most

__device__ unsigned int g_quant_err;

size_t quant_fused_doubles(const sage_params &p) {
    // partial sums (kQuantGridMax + B*H slots of d), then two 32-bit words a head (the count of
    // CTAs that have added their partial, and the flag that mu_K of the head is written)
    return static_cast<size_t>(kQuantGridMax + p.B * p.H) * p.d + static_cast<size_t>(p.B) * p.H;
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned int *p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// INT8 codes of 8 values as bytes: delta > 0 normal, r = fl32(1 / delta).  Packed float32 pairs:
// q = fl32(x r); adding 1.5 2^23 rounds q to the nearest integer k (ties to even) and leaves
// k mod 256 in the low byte of the sum; |q - k| over the eight values decides whether any lies
// near a half-integer, and then all eight take the correctly rounded division.  (Should the code
// generator fuse the product into the addition, k is the rounding of the exact x r, which the
// same test places on the same side of every half-integer.)
// fp16 values of 8 int8 codes (exact)
__device__ __forceinline__ uint4 codes8_to_f16(uint2 c) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t src = i < 2 ? c.x : c.y;
        const int lo = static_cast<int8_t>((src >> (16 * (i & 1))) & 0xFFu);
        const int hi = static_cast<int8_t>((src >> (16 * (i & 1) + 8)) & 0xFFu);
        w[i] = pack_half2(static_cast<float>(lo), static_cast<float>(hi));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool H16 = false>
__device__ __forceinline__ uint2 pack_codes8_rcp(const float (&x)[8], float delta, float r, uint4 *h16 = nullptr) {
    constexpr float kMagic = 12582912.0f;
    const f2 r2{r, r}, m2{kMagic, kMagic};
    f2 t[4], k[4];
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const f2 q = mul2(f2{x[2 * i], x[2 * i + 1]}, r2);
        t[i] = add2(q, m2);
        k[i] = sub2(t[i], m2);
        const f2 e = sub2(q, k[i]);
        dmax = max3f(dmax, fabsf(e.x), fabsf(e.y));
    }
    if (dmax >= 0.499969482421875f) {                  // 1/2 - 2^-15
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            k[i].x = fminf(fmaxf(rintf(__fdiv_rn(x[2 * i], delta)), -127.0f), 127.0f);
            k[i].y = fminf(fmaxf(rintf(__fdiv_rn(x[2 * i + 1], delta)), -127.0f), 127.0f);
            t[i] = add2(k[i], m2);
        }
    }
    if (H16) *h16 = make_uint4(pack_half2(k[0].x, k[0].y), pack_half2(k[1].x, k[1].y), pack_half2(k[2].x, k[2].y),
                               pack_half2(k[3].x, k[3].y));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = __byte_perm(__float_as_uint(t[i].x), __float_as_uint(t[i].y), 0x0040);
    return make_uint2(__byte_perm(w[0], w[1], 0x5410), __byte_perm(w[2], w[3], 0x5410));
}

struct QuantSched {
    int per_z;               // blocks of one tensor: B*H*N/64
    int nz;                  // tensors: 3 (K, Q, V), or 1 (V alone)
    int nA;                  // K-mean blocks: per_z with K-smoothing, else 0
    void *kpart;             // (kQuantGridMax + B*H, d) partial sums: int64 (fp16) or float64 (bf16)
    unsigned int *sync;      // [h] CTAs that added head h's partial, [B*H + h] mu_K of head h
                             // written (zeroed before the launch)
};

// CTA c's share of the K-mean blocks is [c nA / grid, (c + 1) nA / grid); the CTA whose share
// holds block kb, and whether a share holds any block
__device__ __forceinline__ int kmean_owner(long long kb, int nA, int grid) {
    return static_cast<int>(((kb + 1) * grid - 1) / nA);
}
__device__ __forceinline__ bool kmean_share_nonempty(int c, int nA, int grid) {
    return static_cast<long long>(c) * nA / grid < static_cast<long long>(c + 1) * nA / grid;
}
// the CTAs whose shares hold blocks of head h: [c0, c1], and how many of them are non-empty
__device__ __forceinline__ int kmean_contributors(int h, int nb, int nA, int grid, int &c0, int &c1) {
    c0 = kmean_owner(static_cast<long long>(h) * nb, nA, grid);
    c1 = kmean_owner(static_cast<long long>(h) * nb + nb - 1, nA, grid);
    int n = 0;
    for (int c = c0; c <= c1; ++c) n += kmean_share_nonempty(c, nA, grid);
    return n;
}

template <typename T, bool NORM, bool FP8, int D>
__global__ void __launch_bounds__(kQuantThreads, NORM ? 2 : kQuantCtas) quantize_kernel(QuantArgs a, QkNormArgs qn, QuantSched sc) {
    constexpr int kVec = D / 8;                               // threads a row
    constexpr int kRows = kQuantThreads / kVec;               // rows in one pass of the CTA
    constexpr int kIters = 64 / kRows;                        // rows a thread in a block: 4 (d = 128) or 2
    constexpr uint32_t kBlkBytes = 64u * D * sizeof(T);
    constexpr int kStages = kQuantStageBytes / kBlkBytes < kQuantMaxStages ? kQuantStageBytes / kBlkBytes : kQuantMaxStages;
    constexpr bool kHalf = std::is_same<T, __half>::value;
    extern __shared__ __align__(128) uint8_t qsm[];
    __shared__ uint64_t full[kStages];
    __shared__ int4 info[kStages];                            // (z, bh, blk) of the block in each stage
    __shared__ float red[2][8];
    __shared__ float mu_s[D];
    __shared__ int abort_s, fin_s;
    const int tid = threadIdx.x;
    const int N = a.N, nb = N / 64;
    const int grid = gridDim.x, cta = blockIdx.x;
    const int nwork = sc.per_z * sc.nz;
    // this CTA's K-mean share and quantise blocks
    const int a_lo = static_cast<int>(static_cast<long long>(cta) * sc.nA / grid);
    const int a_hi = static_cast<int>(static_cast<long long>(cta + 1) * sc.nA / grid);
    const int nAc = a_hi - a_lo;
    const int mine = nAc + (nwork - cta + grid - 1) / grid;
    double *colsum = reinterpret_cast<double *>(qsm + kStages * kBlkBytes);   // smooth_q / K-mean only
    const int cv = tid % kVec, rg = tid / kVec;

    auto issue = [&](int j) {
        const int s = j % kStages;
        int z, bh, blk;
        if (j < nAc) {
            const int kb = a_lo + j;
            z = 1;
            bh = kb / nb;
            blk = kb - bh * nb;
        } else {
            const int w = cta + (j - nAc) * grid;
            const int zi = w / sc.per_z, rem = w - zi * sc.per_z;
            // K first (still in L2 after the K-mean); measured against K last, the order moves the
            // pass by under 3 % either way (d = 128: K first 1.6 % faster; d = 64: 2.5 % slower)
            z = sc.nz == 1 ? 2 : (zi == 0 ? 1 : (zi == 1 ? 0 : 2));
            bh = rem / nb;
            blk = rem - bh * nb;
        }
        info[s] = make_int4(z, bh, blk, 0);
        const T *base = static_cast<const T *>(z == 0 ? a.Q : (z == 1 ? a.K : a.V));
        mbar_arrive_expect_tx(&full[s], kBlkBytes);
        bulk_load(qsm + s * kBlkBytes, base + (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64) * D,
                  kBlkBytes, &full[s]);
    };
    if (tid == 0) {
        abort_s = 0;
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        for (int j = 0; j < kStages && j < mine; ++j) issue(j);
    }
    __syncthreads();
    // this thread's kIters rows of the block in stage st (16-byte slices, 8 values each)
    auto read_block = [&](int st, float (&x)[kIters][8]) {
        const uint8_t *buf = qsm + st * kBlkBytes;
#pragma unroll
        for (int k = 0; k < kIters; ++k)
            unpack8<T>(*reinterpret_cast<const uint4 *>(buf + ((rg + k * kRows) * D + cv * 8) * sizeof(T)), x[k]);
    };

    int i = 0;
    bool failed = false;
    // ---------------------------------------------------------------- 1. K-mean share
    if (sc.nA > 0) {
        // fp16: v = hi + lo exactly, hi = v rounded to a multiple of 2^-4 (adding 1.5 2^19 rounds
        // there), lo = v - hi a multiple of 2^-24 with |lo| <= 2^-5; sixteen his stay below 2^20
        // (24 bits) and sixteen los below 2^-1 (23 bits), so packed float32 adds sum them exactly,
        // and every sixteen rows they join the int64 total in units of 2^-24.
        long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        f2 hs[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
        f2 ls[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
        Sum3 acc3[8];
        int rows_acc = 0;
        const f2 c2{786432.0f, 786432.0f};                    // 1.5 * 2^19
        auto fold = [&]() {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += (__float2ll_rn(hs[e].x * 16.0f) << 20) + __float2ll_rn(ls[e].x * 16777216.0f);
                acc[2 * e + 1] += (__float2ll_rn(hs[e].y * 16.0f) << 20) + __float2ll_rn(ls[e].y * 16777216.0f);
                hs[e] = f2{0.0f, 0.0f};
                ls[e] = f2{0.0f, 0.0f};
            }
        };
        for (; i < nAc; ++i) {
            const int st = i % kStages;
            const bool ok = mbar_wait_warp(&full[st], (i / kStages) & 1, &abort_s, &g_quant_err, 1);
            const int4 inf = info[st];
            const int bh = inf.y, blk = inf.z;
            float x[kIters][8];
            read_block(st, x);
#pragma unroll
            for (int k = 0; k < kIters; ++k) {
                if (NORM) qk_norm8<T>(x[k], qn.gamma[1], cv * 8, kVec, D, qn.eps);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    if constexpr (kHalf) {
                        const f2 v{x[k][e], x[k][e + 1]};
                        const f2 hi = sub2(add2(v, c2), c2);
                        hs[e / 2] = add2(hs[e / 2], hi);
                        ls[e / 2] = add2(ls[e / 2], sub2(v, hi));
                    } else {
                        acc3[e].add(x[k][e]);
                        acc3[e + 1].add(x[k][e + 1]);
                    }
                }
            }
            if (kHalf && (rows_acc += kIters) == 16) {
                fold();
                rows_acc = 0;
            }
            // every thread has read the stage (and a wait that gave up is seen by all)
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            if (tid == 0 && i + kStages < mine) {
                fence_view_async_shared();
                issue(i + kStages);
            }
            if (blk == nb - 1 || i == nAc - 1) {
                // the end of this CTA's run of head bh: its partial sum, in a fixed order
                if (kHalf) {
                    fold();
                    rows_acc = 0;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if constexpr (kHalf) reinterpret_cast<long long *>(colsum)[tid * 8 + e] = acc[e];
                    else colsum[tid * 8 + e] = acc3[e].value();
                    acc[e] = 0;
                    acc3[e] = Sum3();
                }
                __syncthreads();
                if (tid < D) {
                    const int cvv = tid / 8, ci = tid % 8;
                    if constexpr (kHalf) {
                        long long sum = 0;
                        for (int g = 0; g < kRows; ++g) sum += reinterpret_cast<long long *>(colsum)[(g * kVec + cvv) * 8 + ci];
                        static_cast<long long *>(sc.kpart)[static_cast<size_t>(cta + bh) * D + tid] = sum;
                    } else {
                        double sum = 0.0;
                        for (int g = 0; g < kRows; ++g) sum += colsum[(g * kVec + cvv) * 8 + ci];
                        static_cast<double *>(sc.kpart)[static_cast<size_t>(cta + bh) * D + tid] = sum;
                    }
                }
                __syncthreads();
                // the last CTA to add a partial of head bh writes the head's mean
                int c0, c1;
                const int ncontrib = kmean_contributors(bh, nb, sc.nA, grid, c0, c1);
                if (tid == 0) {
                    __threadfence();
                    fin_s = atomicAdd(&sc.sync[bh], 1u) + 1u == static_cast<unsigned int>(ncontrib);
                }
                __syncthreads();
                if (fin_s) {
                    __threadfence();
                    if (tid < D) {
                        // (with more CTAs than K blocks, some shares are empty and wrote no partial)
                        double sum;
                        if constexpr (kHalf) {
                            long long si = 0;
                            for (int cc = c0; cc <= c1; ++cc)
                                if (kmean_share_nonempty(cc, sc.nA, grid))
                                    si += __ldcg(static_cast<const long long *>(sc.kpart) + static_cast<size_t>(cc + bh) * D + tid);
                            sum = static_cast<double>(si) * 0x1p-24;
                        } else {
                            sum = 0.0;
                            for (int cc = c0; cc <= c1; ++cc)
                                if (kmean_share_nonempty(cc, sc.nA, grid))
                                    sum += __ldcg(static_cast<const double *>(sc.kpart) + static_cast<size_t>(cc + bh) * D + tid);
                        }
                        a.muK[static_cast<size_t>(bh) * D + tid] = static_cast<float>(sum / static_cast<double>(N));
                    }
                    __syncthreads();
                    if (tid == 0) {
                        __threadfence();
                        st_release_gpu(&sc.sync[sc.per_z / nb + bh], 1u);
                    }
                }
            }
        }
    }
    // ---------------------------------------------------------------- 2. smoothing + codes
    for (; i < mine && !failed; ++i) {
        const int st = i % kStages;
        // Every warp waits for the stage itself.  A warp whose bounded wait gave up goes on with
        // whatever the stage holds and posts a negative maximum: after the block-maximum barrier,
        // the one CTA barrier of a block, every warp sees it and the CTA stops before writing.
        bool ok = mbar_wait_warp(&full[st], (i / kStages) & 1, &abort_s, &g_quant_err, 1);
        // (info[st] is rewritten only after the block-maximum barrier below, which every thread
        // reaches after reading it here)
        const int4 inf = info[st];
        const int z = inf.x, bh = inf.y, blk = inf.z;
        const size_t blk_off = (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64) * D;
        float x[kIters][8];
        read_block(st, x);
        const bool norm = NORM && z < 2;               // uniform over the CTA
        if (norm) {
            // selected by value: indexing the parameter's arrays with z would copy them to local memory
            const float *gamma = z == 0 ? qn.gamma[0] : qn.gamma[1];
            float *rnorm = z == 0 ? qn.rnorm[0] : qn.rnorm[1];
            void *xnorm = z == 0 ? qn.xnorm[0] : qn.xnorm[1];
#pragma unroll
            for (int k = 0; k < kIters; ++k) {
                const int r = rg + k * kRows;
                const float rf = qk_norm8<T>(x[k], gamma, cv * 8, kVec, D, qn.eps);
                if (cv == 0) rnorm[static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64 + r] = rf;
                if (xnorm)
                    *reinterpret_cast<uint4 *>(static_cast<T *>(xnorm) + blk_off + static_cast<size_t>(r) * D + cv * 8) =
                        pack8<T>(x[k]);
            }
        }
        // per-channel mean to subtract: mu_K (written before the grid-wide barrier; read through
        // L2), or the block's own mean of Q (float64 sum of its exact values, one rounding of
        // sum / 64)
        bool smooth = false;
        float mu[8];
        if (z == 1 && a.smooth_k) {
            smooth = true;
            // mu_K of head bh is final once the head's flag is up (one lane polls, bounded)
            bool up = true;
            if (lane_id() == 0) {
                const unsigned int *flag = &sc.sync[sc.per_z / nb + bh];
                if (ld_acquire_gpu(flag) == 0u) {
                    const unsigned long long t0 = clock64();
                    while (ld_acquire_gpu(flag) == 0u) {
                        if (*reinterpret_cast<volatile int *>(&abort_s) || clock64() - t0 > SAGE_WAIT_CYCLES) {
                            abort_s = 1;
                            atomicOr(&g_quant_err, 1u | (3u << 8));
                            up = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
            }
            // (the warp barrier orders the lanes' reads of mu_K after lane 0's acquire of the flag;
            // a shuffle alone would let those reads move above the poll)
            __syncwarp();
            up = __shfl_sync(0xffffffffu, up, 0);
            ok = ok && up;
            const float4 *m = reinterpret_cast<const float4 *>(a.muK + static_cast<size_t>(bh) * D + cv * 8);
            *reinterpret_cast<float4 *>(&mu[0]) = __ldcg(m);
            *reinterpret_cast<float4 *>(&mu[4]) = __ldcg(m + 1);
        } else if (z == 1) {
            if (blk == 0 && tid < D) a.muK[static_cast<size_t>(bh) * D + tid] = 0.0f;
        } else if (z == 0 && a.smooth_q) {
            smooth = true;
            // per thread: fp16 values as exact int64 multiples of 2^-24 (no float64 adds, slow on
            // GB300); bf16 in float64
            long long acci[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            double accd[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int k = 0; k < kIters; ++k) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if constexpr (kHalf)
                        acci[e] += half_fixed24(__half_as_ushort(__float2half_rn(x[k][e])));
                    else
                        accd[e] += static_cast<double>(x[k][e]);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if constexpr (kHalf)
                    colsum[tid * 8 + e] = static_cast<double>(acci[e]) * 0x1p-24;
                else
                    colsum[tid * 8 + e] = accd[e];
            }
            __syncthreads();
            if (tid < D) {
                const int cvv = tid / 8, ci = tid % 8;
                double sum = 0.0;
                for (int g = 0; g < kRows; ++g) sum += colsum[(g * kVec + cvv) * 8 + ci];
                const float m = static_cast<float>(sum / 64.0);
                mu_s[tid] = m;
                a.muQ[(static_cast<size_t>(bh) * nb + blk) * D + tid] = m;
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < 8; ++e) mu[e] = mu_s[cv * 8 + e];
        }
        float mxr[kIters];                                    // one running maximum a row: short chains
#pragma unroll
        for (int k = 0; k < kIters; ++k) {
            mxr[k] = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                f2 v{x[k][e], x[k][e + 1]};
                if (smooth) v = sub2(v, f2{mu[e], mu[e + 1]});   // fl32(v - mu), lane by lane
                x[k][e] = v.x;
                x[k][e + 1] = v.y;
                mxr[k] = max3f(mxr[k], fabsf(v.x), fabsf(v.y));
            }
        }
        float mx = mxr[0];
#pragma unroll
        for (int k = 1; k < kIters; ++k) mx = fmaxf(mx, mxr[k]);
        // block maximum; red is double-buffered (its slot is written again two blocks on, after
        // the next block's barrier, which every thread reaches only after reading it here).
        // Non-negative floats order like their bit patterns: one integer maximum over the warp.
        mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
        if ((tid & 31) == 0) red[i & 1][tid >> 5] = ok ? mx : -1.0f;
        __syncthreads();
        float mn = red[i & 1][0];
        mx = mn;
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            mx = fmaxf(mx, red[i & 1][w]);
            mn = fminf(mn, red[i & 1][w]);
        }
        if (mn < 0.0f) {
            failed = true;
            break;
        }
        // every thread has read its values out of this stage: refill it
        if (tid == 0 && i + kStages < mine) {
            fence_view_async_shared();
            issue(i + kStages);
        }
        const float delta = __fdiv_rn(mx, FP8 ? 448.0f : 127.0f);
        int8_t *dst = (z == 0 ? a.Qh : (z == 1 ? a.Kh : a.Vh)) + blk_off + cv * 8;
        // SAGE_FLAG_OPS16: the codes' exact fp16 values too, the tensor cores' operands
        __half *h16 = a.ops16 ? a.ops16 + static_cast<size_t>(z) * sc.per_z * 64 * D + blk_off + cv * 8 : nullptr;
        if (FP8) {
#pragma unroll
            for (int k = 0; k < kIters; ++k) {
                const size_t r = static_cast<size_t>(rg + k * kRows) * D;
                if (h16) {
                    uint4 hv;
                    *reinterpret_cast<uint2 *>(dst + r) = pack_codes8_e4m3_h16(x[k], delta, &hv);
                    *reinterpret_cast<uint4 *>(h16 + r) = hv;
                } else {
                    *reinterpret_cast<uint2 *>(dst + r) = pack_codes8_e4m3(x[k], delta);
                }
            }
        } else if (delta >= 0x1p-126f) {
            const float rcp = __frcp_rn(delta);
            if (h16) {
#pragma unroll
                for (int k = 0; k < kIters; ++k) {
                    const size_t r = static_cast<size_t>(rg + k * kRows) * D;
                    uint4 hv;
                    *reinterpret_cast<uint2 *>(dst + r) = pack_codes8_rcp<true>(x[k], delta, rcp, &hv);
                    *reinterpret_cast<uint4 *>(h16 + r) = hv;
                }
            } else {
#pragma unroll
                for (int k = 0; k < kIters; ++k)
                    *reinterpret_cast<uint2 *>(dst + static_cast<size_t>(rg + k * kRows) * D) = pack_codes8_rcp(x[k], delta, rcp);
            }
        } else {
#pragma unroll
            for (int k = 0; k < kIters; ++k) {
                const size_t r = static_cast<size_t>(rg + k * kRows) * D;
                const uint2 c = pack_codes8(x[k], delta);
                *reinterpret_cast<uint2 *>(dst + r) = c;
                if (h16) *reinterpret_cast<uint4 *>(h16 + r) = codes8_to_f16(c);
            }
        }
        if (tid == 0) {
            float *scale = z == 0 ? a.sQ : (z == 1 ? a.sK : a.sV);
            scale[static_cast<size_t>(bh) * nb + blk] = delta;
        }
    }
    if (failed && tid == 0) {
        // gave up: wait (bounded) for the copies still in flight into this CTA's stages
        for (int j = i; j < i + kStages && j < mine; ++j)
            mbar_wait_drain(&full[j % kStages], (j / kStages) & 1, &g_quant_err, 2);
    }
}

// ---------------------------------------------------------------------------------------------
// NVFP4 ("SageAttention3 ..." (review), eq. (2)-(3) and the NVFP4 row of its format table):
// 1 x 16 blocks, s = e4m3(fl32(max|x| / 6)), codes e2m1(fl32(x / s)), all-zero codes where s = 0.
// Q (z = 0) and K (z = 1), smoothed as for INT8, are blocked along d (a block is the 8 channels
// of two neighbouring lanes); V (z = 2) along the tokens, 16 rows per channel (the block maximum
// through shared-memory atomics on the float bits, which order like the values when >= 0).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_e2m1x8(const float (&x)[8], const float (&s)[8]) {
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = s[2 * i] == 0.0f ? 0.0f : __fdiv_rn(x[2 * i], s[2 * i]);
        const float hi = s[2 * i + 1] == 0.0f ? 0.0f : __fdiv_rn(x[2 * i + 1], s[2 * i + 1]);
        w |= e2m1x2(lo, hi) << (8 * i);
    }
    return w;
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_fp4_kernel(QuantArgs a, Fp4Out o) {
    __shared__ float mu_s[128];
    __shared__ double colsum[256 * 8];
    __shared__ unsigned int vmax[4][128];
    const int blk = blockIdx.x, bh = blockIdx.y, z = blockIdx.z;
    const int d = a.d, N = a.N;
    const T *src = static_cast<const T *>(z == 0 ? a.Q : (z == 1 ? a.K : a.V));
    const int vec_per_row = d / 8;
    const int rows_in_flight = 256 / vec_per_row;
    const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
    const int iters = 64 / rows_in_flight;
    const size_t blk_off = (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64) * d;
    if (z == 2) {
        for (int i = threadIdx.x; i < 4 * 128; i += 256) (&vmax[0][0])[i] = 0u;
    }
    const SmoothIn si{a.kpartial, a.muK, a.muQ, a.ksplits, N, d, a.smooth_k, a.smooth_q};
    const bool smooth = smoothing_mean<T, false>(si, src, z, blk, bh, blk_off, cv, rg, vec_per_row,
                                                  rows_in_flight, iters, nullptr, 0.0f, mu_s, colsum);
    float x[4][8];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        load8(src + blk_off + static_cast<size_t>(rg + it * rows_in_flight) * d + cv * 8, x[it]);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (smooth) x[it][i] = __fsub_rn(x[it][i], mu_s[cv * 8 + i]);
    }
    uint8_t *codes = z == 0 ? o.Qc : (z == 1 ? o.Kc : o.Vc);
    if (z < 2) {
        uint8_t *scales = z == 0 ? o.sQ : o.sK;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            if (it >= iters) break;
            const int r = rg + it * rows_in_flight;
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[it][i]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));       // the block's other lane
            const float sb = e4m3_round_f(__fdiv_rn(m, 6.0f));
            float s8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) s8[i] = sb;
            const size_t row = static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64 + r;
            reinterpret_cast<uint32_t *>(codes + row * (d / 2))[cv] = pack_e2m1x8(x[it], s8);
            if ((cv & 1) == 0) scales[row * (d / 16) + (cv >> 1)] = static_cast<uint8_t>(e4m3x2(sb, 0.0f) & 0xFFu);
        }
        return;
    }
    // V: 16-token blocks per channel
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int g = (rg + it * rows_in_flight) >> 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) atomicMax(&vmax[g][cv * 8 + i], __float_as_uint(fabsf(x[it][i])));
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        const int g = r >> 4;
        float s8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) s8[i] = e4m3_round_f(__fdiv_rn(__uint_as_float(vmax[g][cv * 8 + i]), 6.0f));
        const size_t row = static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64 + r;
        reinterpret_cast<uint32_t *>(codes + row * (d / 2))[cv] = pack_e2m1x8(x[it], s8);
        if ((r & 15) == 0) {
            uint8_t *sv = o.sV + (static_cast<size_t>(bh) * (N / 16) + static_cast<size_t>(blk) * 4 + g) * d + cv * 8;
            uint32_t w0 = 0, w1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w0 |= (e4m3x2(s8[i], 0.0f) & 0xFFu) << (8 * i);
                w1 |= (e4m3x2(s8[4 + i], 0.0f) & 0xFFu) << (8 * i);
            }
            *reinterpret_cast<uint2 *>(sv) = make_uint2(w0, w1);
        }
    }
}

// 16 codes (8 bytes) of one scale block -> 16 fp16 values s * code (exact: at most 6 significant bits)
__global__ void __launch_bounds__(256) widen_fp4_kernel(const uint8_t *__restrict__ codes,
                                                        const uint8_t *__restrict__ scales,
                                                        __half *__restrict__ dst, size_t n16,
                                                        int d, int N, int along_tokens) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const uint2 c = reinterpret_cast<const uint2 *>(codes)[i];
        const uint32_t cw[2] = {c.x, c.y};
        uint32_t sc[8];                                   // 8 fp16 pairs of scales
        if (!along_tokens) {
            const uint32_t b = scales[i];
            const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(b | (b << 8)));
#pragma unroll
            for (int k = 0; k < 8; ++k) sc[k] = h;
        } else {
            // element i*16 .. i*16+15 of row n = (i*16) / d, channels c0 .. c0+15
            const size_t e0 = i * 16;
            const size_t row = e0 / d;                    // (bh * N + n)
            const int c0 = static_cast<int>(e0 % d);
            const size_t bhh = row / N, n = row % N;
            const uint4 sv = *reinterpret_cast<const uint4 *>(scales + (bhh * (N / 16) + n / 16) * d + c0);
            const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sc[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(sw[k] & 0xFFFFu));
                sc[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(sw[k] >> 16));
            }
        }
        uint32_t out[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t byte = (cw[k >> 2] >> (8 * (k & 3))) & 0xFFu;
            out[k] = hmul2(e2m1x2_to_f16x2(byte), sc[k]);
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst) + 2 * i;
        d4[0] = make_uint4(out[0], out[1], out[2], out[3]);
        d4[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
}

// ---------------------------------------------------------------------------------------------
// Attn-QAT fake quantisation ("Attn-QAT: 4-Bit Attention With Quantization-Aware Training",
// technical summary, section 2.2: no smoothing): the NVFP4 quantiser above, Q and K blocked along
// d, V along the tokens, but each value leaves as s * code in the input 16-bit type (exact: at
// most 6 significant bits, magnitudes in [2^-10, 2688]).
// ---------------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ uint4 fake_quant8(const float (&x)[8], const float (&s)[8]) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = s[2 * i] == 0.0f ? 0.0f : __fdiv_rn(x[2 * i], s[2 * i]);
        const float hi = s[2 * i + 1] == 0.0f ? 0.0f : __fdiv_rn(x[2 * i + 1], s[2 * i + 1]);
        const uint32_t h = e2m1x2_to_f16x2(e2m1x2(lo, hi));
        const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&h));
        v[2 * i] = c.x * s[2 * i];                   // exact products
        v[2 * i + 1] = c.y * s[2 * i + 1];
    }
    return pack8<T>(v);
}

template <typename T>
__global__ void __launch_bounds__(256) qat_fake_quant_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                             const T *__restrict__ V, T *__restrict__ Qf,
                                                             T *__restrict__ Kf, T *__restrict__ Vf, int N,
                                                             int d) {
    __shared__ unsigned int vmax[4][128];
    const int blk = blockIdx.x, bh = blockIdx.y, z = blockIdx.z;
    const T *src = z == 0 ? Q : (z == 1 ? K : V);
    T *dst = z == 0 ? Qf : (z == 1 ? Kf : Vf);
    const int vec_per_row = d / 8;
    const int rows_in_flight = 256 / vec_per_row;
    const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
    const int iters = 64 / rows_in_flight;
    const size_t blk_off = (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64) * d;
    if (z == 2) {
        for (int i = threadIdx.x; i < 4 * 128; i += 256) (&vmax[0][0])[i] = 0u;
        __syncthreads();
    }
    float x[4][8];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        load8(src + blk_off + static_cast<size_t>(rg + it * rows_in_flight) * d + cv * 8, x[it]);
    }
    if (z < 2) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            if (it >= iters) break;
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[it][i]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));       // the block's other lane
            const float sb = e4m3_round_f(__fdiv_rn(m, 6.0f));
            float s8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) s8[i] = sb;
            *reinterpret_cast<uint4 *>(dst + blk_off + static_cast<size_t>(rg + it * rows_in_flight) * d + cv * 8) =
                fake_quant8<T>(x[it], s8);
        }
        return;
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int g = (rg + it * rows_in_flight) >> 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) atomicMax(&vmax[g][cv * 8 + i], __float_as_uint(fabsf(x[it][i])));
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        float s8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) s8[i] = e4m3_round_f(__fdiv_rn(__uint_as_float(vmax[r >> 4][cv * 8 + i]), 6.0f));
        *reinterpret_cast<uint4 *>(dst + blk_off + static_cast<size_t>(r) * d + cv * 8) = fake_quant8<T>(x[it], s8);
    }
}

// Attn-QAT backward prologue (section 2.2: the scalar term from dO and the high-precision O'
// alone): D = rowsum(dO o O') with O' in float32, fixed order as in bwd_prologue_kernel, and the
// negated L2 = -fl32(L log2 e).  Thread = (row, 8 channels).
template <typename T>
__global__ void __launch_bounds__(256) qat_bwd_prologue_kernel(const T *__restrict__ dO,
                                                               const float *__restrict__ Op,
                                                               const float *__restrict__ L,
                                                               float *__restrict__ L2,
                                                               float *__restrict__ D, size_t rows,
                                                               int d) {
    const int vec_per_row = d / 8;
    const size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    const size_t row = t / vec_per_row;
    const int cv = static_cast<int>(t % vec_per_row);
    const bool live = row < rows;
    const size_t r = live ? row : rows - 1;
    float x[8], o[8];
    load8(dO + r * d + cv * 8, x);
    const float4 o0 = *reinterpret_cast<const float4 *>(Op + r * d + cv * 8);
    const float4 o1 = *reinterpret_cast<const float4 *>(Op + r * d + cv * 8 + 4);
    o[0] = o0.x; o[1] = o0.y; o[2] = o0.z; o[3] = o0.w;
    o[4] = o1.x; o[5] = o1.y; o[6] = o1.z; o[7] = o1.w;
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) part = __fmaf_rn(x[i], o[i], part);
    for (int o2 = 1; o2 < vec_per_row; o2 <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
    if (live && cv == 0) {
        D[row] = part;
        L2[row] = -__fmul_rn(L[row], kLog2e);
    }
}

// ---------------------------------------------------------------------------------------------
// widen: int8 codes -> integer-valued fp16, or E4M3 codes -> their fp16 values (both exact),
// 16 codes per thread per step
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) widen_e4m3_kernel(const int8_t *__restrict__ src,
                                                         __half *__restrict__ dst, size_t n16) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int4 u = reinterpret_cast<const int4 *>(src)[i];
        const uint32_t w[4] = {static_cast<uint32_t>(u.x), static_cast<uint32_t>(u.y),
                               static_cast<uint32_t>(u.z), static_cast<uint32_t>(u.w)};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            o[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xFFFFu));
            o[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst) + 2 * i;
        d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

__global__ void __launch_bounds__(256) widen_kernel(const int8_t *__restrict__ src,
                                                    __half *__restrict__ dst, size_t n16) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int4 u = reinterpret_cast<const int4 *>(src)[i];
        const uint32_t w[4] = {static_cast<uint32_t>(u.x), static_cast<uint32_t>(u.y),
                               static_cast<uint32_t>(u.z), static_cast<uint32_t>(u.w)};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b0 = static_cast<int8_t>(w[k] & 0xFF), b1 = static_cast<int8_t>((w[k] >> 8) & 0xFF);
            const int b2 = static_cast<int8_t>((w[k] >> 16) & 0xFF), b3 = static_cast<int8_t>(w[k] >> 24);
            __half2 h0 = __halves2half2(__int2half_rn(b0), __int2half_rn(b1));
            __half2 h1 = __halves2half2(__int2half_rn(b2), __int2half_rn(b3));
            o[2 * k] = *reinterpret_cast<uint32_t *>(&h0);
            o[2 * k + 1] = *reinterpret_cast<uint32_t *>(&h1);
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst) + 2 * i;
        d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ---------------------------------------------------------------------------------------------
// backward prologue: D = rowsum(dO o O) (float32, fixed order) and per-block quantisation of dO
// to integer-valued fp16 codes (+ scales; + int8 codes when asked for).
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) bwd_prologue_kernel(BwdPrologueArgs a) {
    __shared__ float red[8];
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int d = a.d, N = a.N;
    const int vec_per_row = d / 8;
    const int rows_in_flight = 256 / vec_per_row;
    const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
    const int iters = 64 / rows_in_flight;
    const size_t blk_off = (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64) * d;
    const T *dO = static_cast<const T *>(a.dO);
    const T *O = static_cast<const T *>(a.O);
    float x[4][8];
    float mx = 0.0f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        float o[8];
        load8(dO + blk_off + static_cast<size_t>(r) * d + cv * 8, x[it]);
        load8(O + blk_off + static_cast<size_t>(r) * d + cv * 8, o);
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            part = __fmaf_rn(x[it][i], o[i], part);
            mx = fmaxf(mx, fabsf(x[it][i]));
        }
        // reduce over the vec_per_row consecutive lanes that share row r (fixed tree order)
        for (int o2 = 1; o2 < vec_per_row; o2 <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
        if (cv == 0) {
            const size_t row = static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64 + r;
            a.D[row] = part;
            a.L2[row] = -__fmul_rn(a.L[row], kLog2e);     // stored negated: -fl32(L log2 e)
        }
    }
    mx = block_max_256(mx, red);
    const float delta = __fdiv_rn(mx, a.fp8 ? 448.0f : 127.0f);
    // INT8 codes of a normal delta: the reciprocal product with the exact tie test (see
    // pack_codes8_rcp), which gives the codes and their fp16 values together
    const bool rcp_path = !a.fp8 && delta >= 0x1p-126f;
    const float rcp = rcp_path ? __frcp_rn(delta) : 0.0f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        const size_t off = blk_off + static_cast<size_t>(r) * d + cv * 8;
        if (rcp_path) {
            uint4 h;
            const uint2 c = pack_codes8_rcp<true>(x[it], delta, rcp, &h);
            *reinterpret_cast<uint4 *>(a.dO16 + off) = h;
            if (a.dOh) *reinterpret_cast<uint2 *>(a.dOh + off) = c;
        } else {
            uint4 h;
            if (a.fp8) (void)pack_codes8_e4m3_h16(x[it], delta, &h);
            else h = pack_codes8_f16(x[it], delta);
            *reinterpret_cast<uint4 *>(a.dO16 + off) = h;
            if (a.dOh) *reinterpret_cast<uint2 *>(a.dOh + off) = pack_codes8(x[it], delta);
        }
    }
    if (threadIdx.x == 0) a.sdO[static_cast<size_t>(bh) * (N / 64) + blk] = delta;
}

// ---------------------------------------------------------------------------------------------
// Q-smoothing bias in log2 units: bias[bh, i, n] = fl32(fl32(sum_c muQ[bh,i,c] * fl32(K[bh,n,c] -
// muK[bh,c])) * sl2), float32 products summed in channel order.
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) qbias_kernel(const T *__restrict__ K,
                                                    const float *__restrict__ muK,
                                                    const float *__restrict__ muQ,
                                                    float *__restrict__ bias, int N, int d,
                                                    float sl2) {
    __shared__ float mq[128];
    __shared__ float mk[128];
    const int i = blockIdx.y, bh = blockIdx.z;
    const int n = blockIdx.x * 256 + threadIdx.x;
    if (threadIdx.x < d) {
        mq[threadIdx.x] = muQ[(static_cast<size_t>(bh) * (N / 64) + i) * d + threadIdx.x];
        mk[threadIdx.x] = muK[static_cast<size_t>(bh) * d + threadIdx.x];
    }
    __syncthreads();
    if (n >= N) return;
    const T *krow = K + (static_cast<size_t>(bh) * N + n) * d;
    float acc = 0.0f;
    for (int c = 0; c < d; c += 8) {
        float v[8];
        load8(krow + c, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = __fmaf_rn(mq[c + k], __fsub_rn(v[k], mk[c + k]), acc);
    }
    bias[(static_cast<size_t>(bh) * (N / 64) + i) * N + n] = __fmul_rn(acc, sl2);
}

// ---------------------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------------------
// SMs of the current device (cached per device; a repeated query is harmless)
static int sm_count() {
    static int cached[16] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 16 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 16) cached[dev] = n;
    return n;
}

template <typename T, bool NORM, bool FP8, int D>
static cudaError_t launch_quantize_k(const sage_params &p, const QuantArgs &a, const QkNormArgs &qn, int nz,
                                     cudaStream_t st) {
    constexpr int blk_bytes = 64 * D * static_cast<int>(sizeof(T));
    constexpr int nstages = kQuantStageBytes / blk_bytes < kQuantMaxStages ? kQuantStageBytes / blk_bytes : kQuantMaxStages;
    const int nb = p.N / 64;
    QuantSched sc;
    sc.per_z = p.B * p.H * nb;
    sc.nz = nz;
    sc.nA = (nz == 3 && p.smooth_k) ? sc.per_z : 0;
    const bool colsum = a.smooth_q || sc.nA > 0;
    const int smem = nstages * blk_bytes + (colsum ? kQuantThreads * 8 * static_cast<int>(sizeof(double)) : 0);
    auto kern = quantize_kernel<T, NORM, FP8, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // CTAs resident together: the K-mean's grid-wide barrier needs every CTA of the launch resident
    static int occ_cache[2] = {0, 0};
    int occ = occ_cache[colsum];
    if (occ <= 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kQuantThreads, smem);
        if (e != cudaSuccess) return e;
        occ_cache[colsum] = occ;
    }
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int want = NORM ? 2 : kQuantCtas;
    int per_sm = occ < want ? occ : want;
    int cap = per_sm * sms;
    if (cap > kQuantGridMax) cap = kQuantGridMax;
    const int nwork = sc.per_z * nz;
    const int grid = nwork < cap ? nwork : cap;
    if (grid <= 0) return cudaSuccess;
    double *scratch = const_cast<double *>(a.kpartial);   // the caller's workspace (written here)
    sc.kpart = scratch;
    sc.sync = nullptr;
    if (sc.nA > 0) {
        if (!a.kpartial || !a.muK) return cudaErrorInvalidValue;
        sc.sync = reinterpret_cast<unsigned int *>(scratch + static_cast<size_t>(kQuantGridMax + p.B * p.H) * D);
        e = cudaMemsetAsync(sc.sync, 0, 2 * sizeof(unsigned int) * static_cast<size_t>(p.B) * p.H, st);
        if (e != cudaSuccess) return e;
        QuantArgs ca = a;
        QkNormArgs cq = qn;
        void *args[] = {&ca, &cq, &sc};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(grid), dim3(kQuantThreads), args,
                                           static_cast<size_t>(smem), st);
    }
    kern<<<grid, kQuantThreads, smem, st>>>(a, qn, sc);
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_quantize_t(const sage_params &p, const QuantArgs &a, const QkNormArgs &qn, int nz, cudaStream_t st) {
    if (a.qk_norm)
        return a.fp8 ? launch_quantize_k<T, true, true, D>(p, a, qn, nz, st)
                     : launch_quantize_k<T, true, false, D>(p, a, qn, nz, st);
    return a.fp8 ? launch_quantize_k<T, false, true, D>(p, a, qn, nz, st)
                 : launch_quantize_k<T, false, false, D>(p, a, qn, nz, st);
}

static cudaError_t launch_quantize_grid(const sage_params &p, const QuantArgs &a, const QkNormArgs &qn,
                                        int nz, cudaStream_t st) {
    if (p.B * p.H * (p.N / 64) == 0) return cudaSuccess;
    if (p.dtype == SAGE_FP16)
        return p.d == 128 ? launch_quantize_t<__half, 128>(p, a, qn, nz, st) : launch_quantize_t<__half, 64>(p, a, qn, nz, st);
    return p.d == 128 ? launch_quantize_t<__nv_bfloat16, 128>(p, a, qn, nz, st)
                      : launch_quantize_t<__nv_bfloat16, 64>(p, a, qn, nz, st);
}

int kmean_splits(const sage_params &p) {
    const int bh = p.B * p.H;
    int s = (8 * 152 + bh - 1) / bh;                   // about eight CTAs per SM
    // at least 16 rows a thread (256 threads, d / 8 of them a row), all of them loaded at once
    const int max_s = static_cast<int>(static_cast<long long>(p.N) * p.d / 32768);
    return s < 1 ? 1 : (s > max_s ? (max_s < 1 ? 1 : max_s) : s);
}

cudaError_t launch_quantize(const sage_params &p, QuantArgs a, cudaStream_t st, const QkNormArgs *qn) {
    QkNormArgs nq{};
    if (qn) nq = *qn;
    if (!a.muK) return cudaErrorInvalidValue;
    return launch_quantize_grid(p, a, nq, 3, st);
}

// V alone (no smoothing applies to V): codes to a.Vh, scales to a.sV
cudaError_t launch_quantize_v(const sage_params &p, QuantArgs a, cudaStream_t st) {
    return launch_quantize_grid(p, a, QkNormArgs{}, 1, st);
}

cudaError_t launch_quantize_fp4(const sage_params &p, QuantArgs a, Fp4Out o, cudaStream_t st) {
    const int bh = p.B * p.H;
    if (p.smooth_k) {
        const int S = a.ksplits;
        const int rows = (p.N + S - 1) / S;
        dim3 g(bh, S);
        double *part = const_cast<double *>(a.kpartial);
        if (p.dtype == SAGE_FP16)
            kmean_partial_kernel<__half, false><<<g, 256, 0, st>>>(static_cast<const __half *>(a.K), part, p.N, p.d, S, rows, nullptr, 0.0f);
        else
            kmean_partial_kernel<__nv_bfloat16, false><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.K), part, p.N, p.d, S, rows, nullptr, 0.0f);
    }
    dim3 g(p.N / 64, bh, 3);
    if (p.dtype == SAGE_FP16)
        quantize_fp4_kernel<__half><<<g, 256, 0, st>>>(a, o);
    else
        quantize_fp4_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(a, o);
    return cudaGetLastError();
}

cudaError_t launch_widen_fp4(const uint8_t *codes, const uint8_t *scales, __half *dst,
                             const sage_params &p, bool along_tokens, cudaStream_t st) {
    const size_t n16 = static_cast<size_t>(p.B) * p.H * p.N * p.d / 16;
    int blocks = static_cast<int>((n16 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    widen_fp4_kernel<<<blocks, 256, 0, st>>>(codes, scales, dst, n16, p.d, p.N, along_tokens ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_qat_fake_quant(const sage_params &p, const void *Q, const void *K, const void *V,
                                  void *Qf, void *Kf, void *Vf, cudaStream_t st) {
    dim3 g(p.N / 64, p.B * p.H, 3);
    if (p.dtype == SAGE_FP16)
        qat_fake_quant_kernel<__half><<<g, 256, 0, st>>>(
            static_cast<const __half *>(Q), static_cast<const __half *>(K), static_cast<const __half *>(V),
            static_cast<__half *>(Qf), static_cast<__half *>(Kf), static_cast<__half *>(Vf), p.N, p.d);
    else
        qat_fake_quant_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(Q), static_cast<const __nv_bfloat16 *>(K),
            static_cast<const __nv_bfloat16 *>(V), static_cast<__nv_bfloat16 *>(Qf),
            static_cast<__nv_bfloat16 *>(Kf), static_cast<__nv_bfloat16 *>(Vf), p.N, p.d);
    return cudaGetLastError();
}

cudaError_t launch_qat_bwd_prologue(const sage_params &p, const void *dO, const float *Op, const float *L,
                                    float *L2, float *D, cudaStream_t st) {
    const size_t rows = static_cast<size_t>(p.B) * p.H * p.N;
    const size_t threads = rows * (p.d / 8);
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    if (p.dtype == SAGE_FP16)
        qat_bwd_prologue_kernel<__half><<<blocks, 256, 0, st>>>(static_cast<const __half *>(dO), Op, L, L2, D, rows, p.d);
    else
        qat_bwd_prologue_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(dO), Op, L,
                                                                       L2, D, rows, p.d);
    return cudaGetLastError();
}

cudaError_t launch_widen(const int8_t *src, __half *dst, size_t n, bool fp8, cudaStream_t st) {
    const size_t n16 = n / 16;
    int blocks = static_cast<int>((n16 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    if (fp8)
        widen_e4m3_kernel<<<blocks, 256, 0, st>>>(src, dst, n16);
    else
        widen_kernel<<<blocks, 256, 0, st>>>(src, dst, n16);
    return cudaGetLastError();
}

cudaError_t launch_bwd_prologue(const sage_params &p, BwdPrologueArgs a, cudaStream_t st) {
    dim3 g(p.N / 64, p.B * p.H);
    if (p.dtype == SAGE_FP16)
        bwd_prologue_kernel<__half><<<g, 256, 0, st>>>(a);
    else
        bwd_prologue_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// QK-norm gradient.  Rows of d / 8 lanes (as in the quantiser), warp-uniform grid-stride loop;
// dg partials per thread, reduced over the CTA's row groups, one float32 reduction per channel.
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) qknorm_bwd_kernel(const T *__restrict__ X,
                                                         const float *__restrict__ g,
                                                         const float *__restrict__ r,
                                                         const float *__restrict__ dY,
                                                         float *__restrict__ dX,
                                                         float *__restrict__ dg, size_t rows, int d) {
    __shared__ float red[256 * 8];
    const int vec_per_row = d / 8;
    const int rows_in_flight = 256 / vec_per_row;
    const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
    float gg[8] = {1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f};
    if (g) {
        *reinterpret_cast<float4 *>(&gg[0]) = *reinterpret_cast<const float4 *>(g + cv * 8);
        *reinterpret_cast<float4 *>(&gg[4]) = *reinterpret_cast<const float4 *>(g + cv * 8 + 4);
    }
    float dga[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const float inv_d = 1.0f / static_cast<float>(d);
    for (size_t b0 = static_cast<size_t>(blockIdx.x) * rows_in_flight; b0 < rows;
         b0 += static_cast<size_t>(gridDim.x) * rows_in_flight) {
        const size_t row = b0 + rg;
        const bool ok = row < rows;
        float x[8] = {0, 0, 0, 0, 0, 0, 0, 0}, dy[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        float rr = 0.0f;
        if (ok) {
            load8(X + row * d + cv * 8, x);
            *reinterpret_cast<float4 *>(&dy[0]) = *reinterpret_cast<const float4 *>(dY + row * d + cv * 8);
            *reinterpret_cast<float4 *>(&dy[4]) = *reinterpret_cast<const float4 *>(dY + row * d + cv * 8 + 4);
            rr = r[row];
        }
        float xh[8], gdy[8], part = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xh[i] = x[i] * rr;
            gdy[i] = gg[i] * dy[i];
            part = fmaf(gdy[i], xh[i], part);
            dga[i] = fmaf(dy[i], xh[i], dga[i]);
        }
        for (int o = 1; o < vec_per_row; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const float m = part * inv_d;
        if (ok) {
            float o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = rr * fmaf(-xh[i], m, gdy[i]);
            *reinterpret_cast<float4 *>(dX + row * d + cv * 8) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4 *>(dX + row * d + cv * 8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
        }
    }
    if (!dg) return;
#pragma unroll
    for (int i = 0; i < 8; ++i) red[threadIdx.x * 8 + i] = dga[i];
    __syncthreads();
    if (threadIdx.x < d) {
        const int c = threadIdx.x, cvv = c / 8, ci = c % 8;
        float sum = 0.0f;
        for (int q = 0; q < rows_in_flight; ++q) sum += red[(q * vec_per_row + cvv) * 8 + ci];
        atomicAdd(dg + c, sum);
    }
}

cudaError_t launch_qknorm_bwd(const sage_params &p, const void *X, const float *g, const float *r,
                              const float *dY, float *dX, float *dg, cudaStream_t st) {
    const size_t rows = static_cast<size_t>(p.B) * p.H * p.N;
    const size_t groups = (rows + (2048 / p.d) - 1) / (2048 / p.d);
    const int blocks = static_cast<int>(groups < 152 * 8 ? groups : 152 * 8);
    if (p.dtype == SAGE_FP16)
        qknorm_bwd_kernel<__half><<<blocks, 256, 0, st>>>(static_cast<const __half *>(X), g, r, dY, dX, dg, rows, p.d);
    else
        qknorm_bwd_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(X), g, r, dY, dX, dg, rows, p.d);
    return cudaGetLastError();
}

cudaError_t launch_qbias(const sage_params &p, const void *K, const float *muK, const float *muQ,
                         float *bias, float sl2, cudaStream_t st) {
    dim3 g((p.N + 255) / 256, p.N / 64, p.B * p.H);
    if (p.dtype == SAGE_FP16)
        qbias_kernel<__half><<<g, 256, 0, st>>>(static_cast<const __half *>(K), muK, muQ, bias, p.N, p.d, sl2);
    else
        qbias_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(K), muK, muQ, bias, p.N, p.d, sl2);
    return cudaGetLastError();
}

unsigned int take_quant_error() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_quant_err, sizeof(v));
    cudaMemcpyToSymbol(g_quant_err, &zero, sizeof(zero));
    return v;
}

}  // namespace sage
