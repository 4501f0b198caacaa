// sage_quant.cu -- smoothing, per-block INT8 quantisation and the streaming helper passes.
//
// "SageBwd: A Trainable Low-bit Attention" (structured summary): prerequisites, INT8 quantisation
// (X^ = round(X / delta), delta = max|X| / 127, per-block granularity aligned with the attention
// tiles) and K-/Q-smoothing (mu_K = mean over tokens of K, K_sm = K - mu_K; mu_Qi = mean over the
// rows of query block i); method steps, forward (2) and backward (1).
// "SageAttention3 ..." (review), eq. (7).
//
// Bit-exact contract (the CPU oracle computes the same thing):
//   block        = 64 tokens x d
//   mu           = float64 sum, float64 divide, one rounding to float32
//   x            = fl32(v - mu)
//   delta        = fl32(max|x| / 127)        (IEEE division, __fdiv_rn)
//   code         = clamp(rint_half_even(fl32(x / delta)), -127, 127), zero block -> delta 0, code 0
// FP8 variant ("SageAttention3 ..." (review), INT8 vs FP8 training): delta = fl32(max|x| / 448)
// and code = E4M3(fl32(x / delta)), round to nearest even, saturating at +-448.
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

// fp16 copies of the E4M3 codes of 8 values
__device__ __forceinline__ uint4 pack_codes8_e4m3_f16(const float (&x)[8], float delta) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = delta == 0.0f ? 0u : e4m3x2_f16x2(__fdiv_rn(x[2 * i], delta), __fdiv_rn(x[2 * i + 1], delta));
    return make_uint4(w[0], w[1], w[2], w[3]);
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

// fp16 value as an exact integer multiple of 2^-24 (the smallest fp16 subnormal): every finite
// fp16 is m 2^-24 (subnormal) or (1024 + m) 2^(e - 25), so the multiple is m or
// (1024 + m) << (e - 1), below 2^40 in magnitude.
__device__ __forceinline__ long long half_fixed24(uint32_t h) {
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    const long long mag = e == 0 ? static_cast<long long>(m) : static_cast<long long>(1024u | m) << (e - 1);
    return (h & 0x8000u) ? -mag : mag;
}

// ---------------------------------------------------------------------------------------------
// a1: partial sums of K over token ranges, exact, one (head, split) per CTA.
// partial[(bh * S + s) * d + c] = sum_{n in split s} K[bh, n, c]
// fp16 input: int64 multiples of 2^-24 (integer adds, far faster than float64 ones here and just
// as exact: a sum of 32768 values stays below 2^55, and any sum below 2^53 is exact in both);
// bf16 input (exponent range of float32): float64.  Both occupy 8 bytes per entry.
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) kmean_partial_kernel(const T *__restrict__ K,
                                                            double *__restrict__ partial, int N,
                                                            int d, int S, int rows_per_split) {
    if constexpr (std::is_same<T, __half>::value) {
        __shared__ long long redi[256 * 8];
        const int bh = blockIdx.x, s = blockIdx.y;
        const int vec_per_row = d / 8;
        const int rows_in_flight = 256 / vec_per_row;
        const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
        const int n0 = s * rows_per_split;
        const int n1 = min(N, n0 + rows_per_split);
        long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        const T *base = K + static_cast<size_t>(bh) * N * d;
        for (int n = n0 + rg; n < n1; n += rows_in_flight) {
            const uint4 w = *reinterpret_cast<const uint4 *>(base + static_cast<size_t>(n) * d + cv * 8);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += half_fixed24(u[i] & 0xFFFFu);
                acc[2 * i + 1] += half_fixed24(u[i] >> 16);
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
        double acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        const T *base = K + static_cast<size_t>(bh) * N * d;
        for (int n = n0 + rg; n < n1; n += rows_in_flight) {
            float v[8];
            load8(base + static_cast<size_t>(n) * d + cv * 8, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += static_cast<double>(v[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) red[threadIdx.x * 8 + i] = acc[i];
        __syncthreads();
        if (threadIdx.x < d) {
            const int c = threadIdx.x, cvv = c / 8, ci = c % 8;
            double sum = 0.0;
            for (int g = 0; g < rows_in_flight; ++g) sum += red[(g * vec_per_row + cvv) * 8 + ci];
            partial[(static_cast<size_t>(bh) * S + s) * d + c] = sum;
        }
    }
}

// ---------------------------------------------------------------------------------------------
// a2: smoothing + per-block quantisation of Q (z=0), K (z=1), V (z=2).  One 64 x d block per CTA.
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) quantize_kernel(QuantArgs a) {
    __shared__ float red[8];
    __shared__ float mu_s[128];
    __shared__ double colsum[256 * 8];
    const int blk = blockIdx.x, bh = blockIdx.y, z = blockIdx.z + a.z_base;
    const int d = a.d, N = a.N;
    const T *src = static_cast<const T *>(z == 0 ? a.Q : (z == 1 ? a.K : a.V));
    int8_t *dst = z == 0 ? a.Qh : (z == 1 ? a.Kh : a.Vh);
    float *scale = z == 0 ? a.sQ : (z == 1 ? a.sK : a.sV);
    const int vec_per_row = d / 8;
    const int rows_in_flight = 256 / vec_per_row;
    const int cv = threadIdx.x % vec_per_row, rg = threadIdx.x / vec_per_row;
    const int iters = 64 / rows_in_flight;            // 4 for d = 128, 2 for d = 64
    const size_t blk_off = (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * 64) * d;

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
        double acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int it = 0; it < iters; ++it) {
            const int r = rg + it * rows_in_flight;
            float v[8];
            load8(src + blk_off + static_cast<size_t>(r) * d + cv * 8, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += static_cast<double>(v[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) colsum[threadIdx.x * 8 + i] = acc[i];
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

    float x[4][8];
    float mx = 0.0f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        load8(src + blk_off + static_cast<size_t>(r) * d + cv * 8, x[it]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (smooth) x[it][i] = __fsub_rn(x[it][i], mu_s[cv * 8 + i]);
            mx = fmaxf(mx, fabsf(x[it][i]));
        }
    }
    mx = block_max_256(mx, red);
    const float delta = __fdiv_rn(mx, a.fp8 ? 448.0f : 127.0f);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        *reinterpret_cast<uint2 *>(dst + blk_off + static_cast<size_t>(r) * d + cv * 8) =
            a.fp8 ? pack_codes8_e4m3(x[it], delta) : pack_codes8(x[it], delta);
    }
    if (threadIdx.x == 0) scale[static_cast<size_t>(bh) * (N / 64) + blk] = delta;
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
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        if (it >= iters) break;
        const int r = rg + it * rows_in_flight;
        *reinterpret_cast<uint4 *>(a.dO16 + blk_off + static_cast<size_t>(r) * d + cv * 8) =
            a.fp8 ? pack_codes8_e4m3_f16(x[it], delta) : pack_codes8_f16(x[it], delta);
        if (a.dOh)
            *reinterpret_cast<uint2 *>(a.dOh + blk_off + static_cast<size_t>(r) * d + cv * 8) =
                pack_codes8(x[it], delta);
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
int kmean_splits(const sage_params &p) {
    const int bh = p.B * p.H;
    int s = (2 * 152 + bh - 1) / bh;
    const int max_s = p.N / 64;
    return s < 1 ? 1 : (s > max_s ? max_s : s);
}

cudaError_t launch_quantize(const sage_params &p, QuantArgs a, cudaStream_t st) {
    const int bh = p.B * p.H;
    if (p.smooth_k) {
        const int S = a.ksplits;
        const int rows = (p.N + S - 1) / S;
        dim3 g(bh, S);
        if (p.dtype == SAGE_FP16)
            kmean_partial_kernel<__half><<<g, 256, 0, st>>>(static_cast<const __half *>(a.K), const_cast<double *>(a.kpartial), p.N, p.d, S, rows);
        else
            kmean_partial_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.K), const_cast<double *>(a.kpartial), p.N, p.d, S, rows);
    }
    dim3 g(p.N / 64, bh, 3);
    if (p.dtype == SAGE_FP16)
        quantize_kernel<__half><<<g, 256, 0, st>>>(a);
    else
        quantize_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// V alone (no smoothing applies to V): codes to a.Vh, scales to a.sV
cudaError_t launch_quantize_v(const sage_params &p, QuantArgs a, cudaStream_t st) {
    a.z_base = 2;
    dim3 g(p.N / 64, p.B * p.H, 1);
    if (p.dtype == SAGE_FP16)
        quantize_kernel<__half><<<g, 256, 0, st>>>(a);
    else
        quantize_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(a);
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

cudaError_t launch_qbias(const sage_params &p, const void *K, const float *muK, const float *muQ,
                         float *bias, float sl2, cudaStream_t st) {
    dim3 g((p.N + 255) / 256, p.N / 64, p.B * p.H);
    if (p.dtype == SAGE_FP16)
        qbias_kernel<__half><<<g, 256, 0, st>>>(static_cast<const __half *>(K), muK, muQ, bias, p.N, p.d, sl2);
    else
        qbias_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(K), muK, muQ, bias, p.N, p.d, sl2);
    return cudaGetLastError();
}

}  // namespace sage
