// Row kernels of the block backward pass ("RankMixer 详解（1）" section 5.2):
// the LN1 recompute that feeds the FFN recompute, the LN2 backward, the LN1
// backward fused with the mixing transpose (dX = dY + P^T dY), fixed-order
// reductions of the per-block parameter-gradient partials, and the mean
// pool's backward.
//
// The LayerNorm input gradient of a row with input r, output gradient g and
// affine gamma is
//   dr_j = (q_j - mean(q) - rhat_j mean(q rhat)) / sqrt(var + eps),  q = g gamma,
// with rhat the normalised row; the affine parameters receive g rhat and g.
// Every kernel first reduces a row per warp (statistics), then walks the
// columns with one thread per column, so the parameter-gradient sums over rows
// run in a fixed order inside a thread (deterministic for a given launch shape).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rm_common.cuh"
#include "rm_train.h"
#include "rm_train_math.cuh"

namespace rm {
namespace {

constexpr int kLn2Threads = 256;
constexpr int kLn2Chunk = 8;                 // rows staged in shared memory per step (one per warp)
constexpr int kLn2MaxCols = 3072 / kLn2Threads;
constexpr int kLn1Threads = 256;
constexpr int kLn1MaxCols = 3072 / kLn1Threads;
constexpr int kRowMaxT = 128;

// k / q for 0 <= k < 2^16 by a multiply-high: with m = ceil(2^32 / q) the
// error of k m / 2^32 against k / q stays below 2^-16 < 1 / q, so the floor
// is exact for 2 <= q < 2^16 (checked exhaustively on the host for q <= 3072);
// q = 1 is the identity (m = 0 marks it).
struct QDiv {
    uint32_t q, m;
    __device__ __forceinline__ int div(int k) const { return m == 0 ? k : (int)__umulhi((uint32_t)k, m); }
};

QDiv make_qdiv(int q) {
    QDiv d;
    d.q = (uint32_t)q;
    d.m = q == 1 ? 0u : (uint32_t)((((uint64_t)1 << 32) + (uint64_t)q - 1) / (uint64_t)q);
    return d;
}

// After a bounded wait gave up: wait (again bounded, ignoring the abort flag)
// for the bulk copies still counted on `bar`, so that none lands in shared
// memory after the CTA has exited.
__device__ __forceinline__ void drain_copies(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return;
    }
}

// Element k of the residual row y = Mix(X)[t] + X[t] of one sample:
// Mix(X)[t][c q + r] = X[c][t q + r].
template <typename Tx>
__device__ __forceinline__ float mixed_row_elem(const Tx* __restrict__ Xb, int t, int k, QDiv qd, int D) {
    const int c = qd.div(k), r = k - c * (int)qd.q;
    return to_f32(Xb[(size_t)c * D + (size_t)t * qd.q + r]) + to_f32(Xb[(size_t)t * D + k]);
}

// ---- LN1 recompute ---------------------------------------------------------------
// One warp per row (b, t): y = Mix(X)[t] + X[t] (two loads per element, no
// division), its mean and rstd with shifted sums, then S = gamma1 yhat + beta1
// (operand type), yhat itself (Tyh) and rstd for the LN1 backward.
template <typename Tx, typename Top, typename Tyh>
__global__ void __launch_bounds__(256)
ln1_recompute_kernel(const Tx* __restrict__ X, Top* __restrict__ S, Tyh* __restrict__ Yh, float* __restrict__ rstd_out,
                     const float* __restrict__ g1, const float* __restrict__ be1, int B, int T, int D, int Bcap,
                     float eps, QDiv qd) {
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * T;
    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += (long long)gridDim.x * 8) {
        const int b = (int)(row / T), t = (int)(row - (long long)b * T);
        const Tx* Xb = X + (size_t)b * T * D;
        const float shift = mixed_row_elem(Xb, t, 0, qd, D);
        float s1 = 0.f, s2 = 0.f;
        for (int k = lane; k < D; k += 32) {
            const float d = mixed_row_elem(Xb, t, k, qd, D) - shift;
            s1 += d;
            s2 = fmaf(d, d, s2);
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        const float dm = s1 / (float)D;
        const float mean = shift + dm;
        const float rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
        const size_t o = ((size_t)t * Bcap + b) * D;
        for (int k = lane; k < D; k += 32) {
            const float yh = (mixed_row_elem(Xb, t, k, qd, D) - mean) * rstd;
            S[o + k] = from_f32<Top>(fmaf(g1[k], yh, be1[k]));
            Yh[o + k] = from_f32<Tyh>(yh);
        }
        if (lane == 0) rstd_out[(size_t)t * Bcap + b] = rstd;
    }
}

// The same on column pairs (q even): lane l takes k = 2 l + 64 i, both
// elements of a pair in the same head chunk, so each load and store moves two.
template <typename T>
__device__ __forceinline__ float2 ld_pair(const T* p);
template <>
__device__ __forceinline__ float2 ld_pair<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
template <>
__device__ __forceinline__ float2 ld_pair<float>(const float* p) {
    return *reinterpret_cast<const float2*>(p);
}
template <typename T>
__device__ __forceinline__ void st_pair(T* p, float a, float b);
template <>
__device__ __forceinline__ void st_pair<__half>(__half* p, float a, float b) {
    *reinterpret_cast<__half2*>(p) = __floats2half2_rn(sat_f16(a), sat_f16(b));
}
template <>
__device__ __forceinline__ void st_pair<float>(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
}

template <typename Tx, typename Top, typename Tyh>
__global__ void __launch_bounds__(256)
ln1_recompute_pair_kernel(const Tx* __restrict__ X, Top* __restrict__ S, Tyh* __restrict__ Yh,
                          float* __restrict__ rstd_out, const float* __restrict__ g1, const float* __restrict__ be1,
                          int B, int T, int D, int Bcap, float eps, QDiv qd) {
    const int lane = threadIdx.x & 31;
    const int q = (int)qd.q;
    const long long rows = (long long)B * T;
    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += (long long)gridDim.x * 8) {
        const int b = (int)(row / T), t = (int)(row - (long long)b * T);
        const Tx* Xb = X + (size_t)b * T * D;
        const Tx* Xt = Xb + (size_t)t * D;
        const float shift = to_f32(Xb[(size_t)t * q]) + to_f32(Xt[0]);
        float s1 = 0.f, s2 = 0.f;
        for (int k = 2 * lane; k < D; k += 64) {
            const int c = qd.div(k), r = k - c * q;
            const float2 m = ld_pair<Tx>(Xb + (size_t)c * D + (size_t)t * q + r);
            const float2 x = ld_pair<Tx>(Xt + k);
            const float d0 = m.x + x.x - shift, d1 = m.y + x.y - shift;
            s1 += d0 + d1;
            s2 = fmaf(d0, d0, fmaf(d1, d1, s2));
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        const float dm = s1 / (float)D;
        const float mean = shift + dm;
        const float rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
        const size_t o = ((size_t)t * Bcap + b) * D;
        for (int k = 2 * lane; k < D; k += 64) {
            const int c = qd.div(k), r = k - c * q;
            const float2 m = ld_pair<Tx>(Xb + (size_t)c * D + (size_t)t * q + r);
            const float2 x = ld_pair<Tx>(Xt + k);
            const float2 ga = *reinterpret_cast<const float2*>(g1 + k);
            const float2 be = *reinterpret_cast<const float2*>(be1 + k);
            const float y0 = (m.x + x.x - mean) * rstd, y1 = (m.y + x.y - mean) * rstd;
            st_pair<Top>(S + o + k, fmaf(ga.x, y0, be.x), fmaf(ga.y, y1, be.y));
            st_pair<Tyh>(Yh + o + k, y0, y1);
        }
        if (lane == 0) rstd_out[(size_t)t * Bcap + b] = rstd;
    }
}

// The same with the sample staged in shared memory: a CTA of 1024 threads
// loads sample b's T x D inputs once with 16-byte loads, then a warp per token
// row runs both passes from there (the pair kernel above reads each sample's
// rows about four times through L2).  Same arithmetic in the same order.
constexpr int kLn1RecThreads = 1024;
constexpr size_t kLn1RecSmemLimit = 200 * 1024;

template <typename Tx, typename Top, typename Tyh>
__global__ void __launch_bounds__(kLn1RecThreads, 1)
ln1_recompute_staged_kernel(const Tx* __restrict__ X, Top* __restrict__ S, Tyh* __restrict__ Yh,
                            float* __restrict__ rstd_out, const float* __restrict__ g1, const float* __restrict__ be1,
                            int B, int T, int D, int Bcap, float eps, QDiv qd) {
    extern __shared__ uint4 xs4[];
    const Tx* xs = reinterpret_cast<const Tx*>(xs4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int q = (int)qd.q;
    const int n16 = (int)((size_t)T * D * sizeof(Tx) / 16);
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        __syncthreads();                       // the previous sample's rows are no longer read
        const uint4* src = reinterpret_cast<const uint4*>(X + (size_t)b * T * D);
#pragma unroll 4
        for (int i = threadIdx.x; i < n16; i += blockDim.x) xs4[i] = __ldg(src + i);
        __syncthreads();
        for (int t = warp; t < T; t += nw) {
            const Tx* Xt = xs + (size_t)t * D;
            const float shift = to_f32(xs[(size_t)t * q]) + to_f32(Xt[0]);
            float s1 = 0.f, s2 = 0.f;
            for (int k = 2 * lane; k < D; k += 64) {
                const int c = qd.div(k), r = k - c * q;
                const float2 m = ld_pair<Tx>(xs + (size_t)c * D + (size_t)t * q + r);
                const float2 x = ld_pair<Tx>(Xt + k);
                const float d0 = m.x + x.x - shift, d1 = m.y + x.y - shift;
                s1 += d0 + d1;
                s2 = fmaf(d0, d0, fmaf(d1, d1, s2));
            }
            s1 = warp_sum(s1);
            s2 = warp_sum(s2);
            const float dm = s1 / (float)D;
            const float mean = shift + dm;
            const float rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
            const size_t o = ((size_t)t * Bcap + b) * D;
            for (int k = 2 * lane; k < D; k += 64) {
                const int c = qd.div(k), r = k - c * q;
                const float2 m = ld_pair<Tx>(xs + (size_t)c * D + (size_t)t * q + r);
                const float2 x = ld_pair<Tx>(Xt + k);
                const float2 ga = *reinterpret_cast<const float2*>(g1 + k);
                const float2 be = *reinterpret_cast<const float2*>(be1 + k);
                const float y0 = (m.x + x.x - mean) * rstd, y1 = (m.y + x.y - mean) * rstd;
                st_pair<Top>(S + o + k, fmaf(ga.x, y0, be.x), fmaf(ga.y, y1, be.y));
                st_pair<Tyh>(Yh + o + k, y0, y1);
            }
            if (lane == 0) rstd_out[(size_t)t * Bcap + b] = rstd;
        }
    }
}

// ---- LN2 backward ----------------------------------------------------------------
// Grid (nbx, T): CTA (x, t) walks its share of token t's rows in chunks of 8,
// each chunk staged in shared memory (Z and G rows) so both passes read it
// from there: a warp per row for the statistics (mean, rstd, mean(q),
// mean(q zhat), q = G gamma2), then a thread per column for dZ and the
// column sums of dZ, G zhat and G, kept in registers across the CTA's rows.
template <typename Tz>
__global__ void __launch_bounds__(kLn2Threads)
ln2_backward_kernel(const Tz* __restrict__ Z, const float* __restrict__ G, const float* __restrict__ g2,
                    float* __restrict__ dZ, float* __restrict__ part_db2, float* __restrict__ part_dg2,
                    float* __restrict__ part_dbe2, float* __restrict__ part_max, int B, int T, int D, int Bcap,
                    float eps, int rows_per_cta) {
    extern __shared__ float4 smem4[];
    float4* st = smem4;                                            // [kLn2Chunk]
    float* gs = reinterpret_cast<float*>(smem4 + kLn2Chunk);       // [kLn2Chunk][D]
    Tz* zs = reinterpret_cast<Tz*>(gs + (size_t)kLn2Chunk * D);    // [kLn2Chunk][D]
    __shared__ float wmax[kLn2Threads / 32];
    const int t = blockIdx.y, bx = blockIdx.x, nbx = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b_begin = bx * rows_per_cta;
    const int b_end = min(B, b_begin + rows_per_cta);
    float adb[kLn2MaxCols], adg[kLn2MaxCols], adbe[kLn2MaxCols];
#pragma unroll
    for (int c = 0; c < kLn2MaxCols; ++c) adb[c] = adg[c] = adbe[c] = 0.f;
    float amax = 0.f;
    const bool vec = (D * sizeof(Tz)) % 16 == 0;
    for (int b0 = b_begin; b0 < b_end; b0 += kLn2Chunk) {
        const int nrows = min(kLn2Chunk, b_end - b0);
        __syncthreads();                       // the previous chunk is done with the staged rows
        if (vec) {
            const int zq = D * (int)sizeof(Tz) / 16, gq = D / 4;
            for (int i = threadIdx.x; i < nrows * zq; i += kLn2Threads) {
                const int rr = i / zq, j = i - rr * zq;
                reinterpret_cast<uint4*>(zs + (size_t)rr * D)[j] =
                    __ldg(reinterpret_cast<const uint4*>(Z + ((size_t)t * Bcap + b0 + rr) * D) + j);
            }
            for (int i = threadIdx.x; i < nrows * gq; i += kLn2Threads) {
                const int rr = i / gq, j = i - rr * gq;
                reinterpret_cast<float4*>(gs + (size_t)rr * D)[j] =
                    __ldg(reinterpret_cast<const float4*>(G + ((size_t)(b0 + rr) * T + t) * D) + j);
            }
        } else {
            for (int i = threadIdx.x; i < nrows * D; i += kLn2Threads) {
                const int rr = i / D, k = i - rr * D;
                zs[(size_t)rr * D + k] = Z[((size_t)t * Bcap + b0 + rr) * D + k];
                gs[(size_t)rr * D + k] = G[((size_t)(b0 + rr) * T + t) * D + k];
            }
        }
        __syncthreads();
        if (warp < nrows) {
            const Tz* z = zs + (size_t)warp * D;
            const float* gr = gs + (size_t)warp * D;
            const float shift = to_f32(z[0]);
            float s1 = 0.f, s2 = 0.f;
            for (int k = lane; k < D; k += 32) {
                const float d = to_f32(z[k]) - shift;
                s1 += d;
                s2 = fmaf(d, d, s2);
            }
            s1 = warp_sum(s1);
            s2 = warp_sum(s2);
            const float dm = s1 / (float)D;
            const float mean = shift + dm;
            const float rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
            float mq = 0.f, mqz = 0.f;
            for (int k = lane; k < D; k += 32) {
                const float qk = gr[k] * g2[k];
                mq += qk;
                mqz = fmaf(qk, (to_f32(z[k]) - mean) * rstd, mqz);
            }
            mq = warp_sum(mq);
            mqz = warp_sum(mqz);
            if (lane == 0) st[warp] = make_float4(mean, rstd, mq / (float)D, mqz / (float)D);
        }
        __syncthreads();
        for (int i = 0; i < nrows; ++i) {
            const float4 s = st[i];
            float* dz = dZ + ((size_t)t * Bcap + b0 + i) * D;
#pragma unroll
            for (int c = 0; c < kLn2MaxCols; ++c) {
                const int k = threadIdx.x + c * kLn2Threads;
                if (k < D) {
                    const float zh = (to_f32(zs[(size_t)i * D + k]) - s.x) * s.y;
                    const float gk = gs[(size_t)i * D + k];
                    const float d = (gk * g2[k] - s.z - zh * s.w) * s.y;
                    dz[k] = d;
                    amax = fmaxf(amax, fabsf(d));
                    adb[c] += d;
                    adg[c] = fmaf(gk, zh, adg[c]);
                    adbe[c] += gk;
                }
            }
        }
    }
    const size_t prow = ((size_t)t * nbx + bx) * D;
#pragma unroll
    for (int c = 0; c < kLn2MaxCols; ++c) {
        const int k = threadIdx.x + c * kLn2Threads;
        if (k < D) {
            part_db2[prow + k] = adb[c];
            part_dg2[prow + k] = adg[c];
            part_dbe2[prow + k] = adbe[c];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < kLn2Threads / 32; ++w) m = fmaxf(m, wmax[w]);
        part_max[(size_t)t * nbx + bx] = m;
    }
}

// The same for D a multiple of 4: one pass per row for the statistics (4
// columns per lane step; mean(q zhat) = rstd (sum q (z - shift) - (mean -
// shift) sum q) / D with the row's first value as the shift), and column
// pairs per thread in the second phase.
template <typename Tz>
__device__ __forceinline__ float4 ld4_any(const Tz* p);
template <>
__device__ __forceinline__ float4 ld4_any<__half>(const __half* p) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <>
__device__ __forceinline__ float4 ld4_any<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <typename Tz>
__device__ __forceinline__ float2 ld2_any(const Tz* p);
template <>
__device__ __forceinline__ float2 ld2_any<__half>(const __half* p) {
    return __half22float2(*reinterpret_cast<const __half2*>(p));
}
template <>
__device__ __forceinline__ float2 ld2_any<float>(const float* p) {
    return *reinterpret_cast<const float2*>(p);
}

constexpr int kLn2MaxPairs = 3072 / 2 / kLn2Threads;

template <typename Tz>
__global__ void __launch_bounds__(kLn2Threads, 3)
ln2_backward_vec_kernel(const Tz* __restrict__ Z, const float* __restrict__ G, const float* __restrict__ g2,
                        float* __restrict__ dZ, float* __restrict__ part_db2, float* __restrict__ part_dg2,
                        float* __restrict__ part_dbe2, float* __restrict__ part_max, int B, int T, int D, int Bcap,
                        float eps, int rows_per_cta) {
    extern __shared__ float4 smem4[];
    float4* st = smem4;                                            // [kLn2Chunk]
    float* gs = reinterpret_cast<float*>(smem4 + kLn2Chunk);       // [kLn2Chunk][D]
    Tz* zs = reinterpret_cast<Tz*>(gs + (size_t)kLn2Chunk * D);    // [kLn2Chunk][D]
    __shared__ float wmax[kLn2Threads / 32];
    const int t = blockIdx.y, bx = blockIdx.x, nbx = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b_begin = bx * rows_per_cta;
    const int b_end = min(B, b_begin + rows_per_cta);
    const int npairs = D / 2;
    float2 adb[kLn2MaxPairs], adg[kLn2MaxPairs], adbe[kLn2MaxPairs];
#pragma unroll
    for (int j = 0; j < kLn2MaxPairs; ++j) adb[j] = adg[j] = adbe[j] = make_float2(0.f, 0.f);
    float amax = 0.f;
    const int zq = D * (int)sizeof(Tz) / 16, gq = D / 4;
    for (int b0 = b_begin; b0 < b_end; b0 += kLn2Chunk) {
        const int nrows = min(kLn2Chunk, b_end - b0);
        __syncthreads();                       // the previous chunk is done with the staged rows
        for (int i = threadIdx.x; i < nrows * zq; i += kLn2Threads) {
            const int rr = i / zq, j = i - rr * zq;
            reinterpret_cast<uint4*>(zs + (size_t)rr * D)[j] =
                __ldg(reinterpret_cast<const uint4*>(Z + ((size_t)t * Bcap + b0 + rr) * D) + j);
        }
        for (int i = threadIdx.x; i < nrows * gq; i += kLn2Threads) {
            const int rr = i / gq, j = i - rr * gq;
            reinterpret_cast<float4*>(gs + (size_t)rr * D)[j] =
                __ldg(reinterpret_cast<const float4*>(G + ((size_t)(b0 + rr) * T + t) * D) + j);
        }
        __syncthreads();
        if (warp < nrows) {
            const Tz* z = zs + (size_t)warp * D;
            const float* gr = gs + (size_t)warp * D;
            const float shift = to_f32(z[0]);
            float s1 = 0.f, s2 = 0.f, sq = 0.f, sqz = 0.f;
            for (int k = 4 * lane; k < D; k += 128) {
                const float4 zz = ld4_any<Tz>(z + k);
                const float4 gg = *reinterpret_cast<const float4*>(gr + k);
                const float4 ga = __ldg(reinterpret_cast<const float4*>(g2 + k));
                const float d0 = zz.x - shift, d1 = zz.y - shift, d2 = zz.z - shift, d3 = zz.w - shift;
                const float q0 = gg.x * ga.x, q1 = gg.y * ga.y, q2 = gg.z * ga.z, q3 = gg.w * ga.w;
                s1 += (d0 + d1) + (d2 + d3);
                s2 = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, s2))));
                sq += (q0 + q1) + (q2 + q3);
                sqz = fmaf(q0, d0, fmaf(q1, d1, fmaf(q2, d2, fmaf(q3, d3, sqz))));
            }
            s1 = warp_sum(s1);
            s2 = warp_sum(s2);
            sq = warp_sum(sq);
            sqz = warp_sum(sqz);
            const float dm = s1 / (float)D;
            const float rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
            if (lane == 0)
                st[warp] = make_float4(shift + dm, rstd, sq / (float)D, rstd * (sqz - dm * sq) / (float)D);
        }
        __syncthreads();
#pragma unroll 4
        for (int i = 0; i < nrows; ++i) {
            const float4 s = st[i];
            float* dz = dZ + ((size_t)t * Bcap + b0 + i) * D;
#pragma unroll
            for (int j = 0; j < kLn2MaxPairs; ++j) {
                const int pidx = threadIdx.x + j * kLn2Threads;
                if (pidx < npairs) {
                    const int k = 2 * pidx;
                    const float2 zz = ld2_any<Tz>(zs + (size_t)i * D + k);
                    const float2 gk = *reinterpret_cast<const float2*>(gs + (size_t)i * D + k);
                    const float2 ga = __ldg(reinterpret_cast<const float2*>(g2 + k));
                    const float zh0 = (zz.x - s.x) * s.y, zh1 = (zz.y - s.x) * s.y;
                    float2 d;
                    d.x = (gk.x * ga.x - s.z - zh0 * s.w) * s.y;
                    d.y = (gk.y * ga.y - s.z - zh1 * s.w) * s.y;
                    *reinterpret_cast<float2*>(dz + k) = d;
                    amax = fmaxf(amax, fmaxf(fabsf(d.x), fabsf(d.y)));
                    adb[j].x += d.x;
                    adb[j].y += d.y;
                    adg[j].x = fmaf(gk.x, zh0, adg[j].x);
                    adg[j].y = fmaf(gk.y, zh1, adg[j].y);
                    adbe[j].x += gk.x;
                    adbe[j].y += gk.y;
                }
            }
        }
    }
    const size_t prow = ((size_t)t * nbx + bx) * D;
#pragma unroll
    for (int j = 0; j < kLn2MaxPairs; ++j) {
        const int pidx = threadIdx.x + j * kLn2Threads;
        if (pidx < npairs) {
            *reinterpret_cast<float2*>(part_db2 + prow + 2 * pidx) = adb[j];
            *reinterpret_cast<float2*>(part_dg2 + prow + 2 * pidx) = adg[j];
            *reinterpret_cast<float2*>(part_dbe2 + prow + 2 * pidx) = adbe[j];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < kLn2Threads / 32; ++w) m = fmaxf(m, wmax[w]);
        part_max[(size_t)t * nbx + bx] = m;
    }
}

// Double-buffered variant (D a multiple of 8, two chunks fit in shared
// memory): a chunk is CH rows of one token; while the CTA computes chunk i
// from one buffer, chunk i + 1 arrives in the other by bulk copies (the CH Z
// rows are one contiguous block; the CH G rows are T D floats apart),
// completion counted on that buffer's mbarrier with a bounded wait.  CH = 4
// keeps a CTA at 74 KB for the 1B width, so three share an SM and keep three
// chunks in flight.
template <typename Tz, int CH>
__global__ void __launch_bounds__(kLn2Threads)
ln2_backward_db_kernel(const Tz* __restrict__ Z, const float* __restrict__ G, const float* __restrict__ g2,
                       float* __restrict__ dZ, float* __restrict__ part_db2, float* __restrict__ part_dg2,
                       float* __restrict__ part_dbe2, float* __restrict__ part_max, int B, int T, int D, int Bcap,
                       float eps, int rows_per_cta, int* err, unsigned long long timeout_ns) {
    extern __shared__ float4 smem4[];
    float4* st = smem4;                                            // [CH]
    float* gbuf = reinterpret_cast<float*>(smem4 + CH);     // 2 x [CH][D]
    Tz* zbuf = reinterpret_cast<Tz*>(gbuf + 2 * (size_t)CH * D);   // 2 x [CH][D]
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int s_abort;
    __shared__ float wmax[kLn2Threads / 32];
    const int t = blockIdx.y, bx = blockIdx.x, nbx = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b_begin = bx * rows_per_cta;
    const int b_end = min(B, b_begin + rows_per_cta);
    const int npairs = D / 2;
    float2 adb[kLn2MaxPairs], adg[kLn2MaxPairs], adbe[kLn2MaxPairs];
#pragma unroll
    for (int j = 0; j < kLn2MaxPairs; ++j) adb[j] = adg[j] = adbe[j] = make_float2(0.f, 0.f);
    float amax = 0.f;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int chunk, int buf) {     // thread 0: chunk `chunk` of this CTA into buffer `buf`
        const int b0 = b_begin + chunk * CH;
        const int nrows = min(CH, b_end - b0);
        const uint32_t bar = smem_u32(&bars[buf]);
        const uint32_t zbytes = (uint32_t)(nrows * D * sizeof(Tz)), gbytes = (uint32_t)(D * sizeof(float));
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, zbytes + gbytes * (uint32_t)nrows);
        bulk_copy_g2s(smem_u32(zbuf + (size_t)buf * CH * D), Z + ((size_t)t * Bcap + b0) * D, zbytes, bar);
        for (int r = 0; r < nrows; ++r)
            bulk_copy_g2s(smem_u32(gbuf + ((size_t)buf * CH + r) * D), G + ((size_t)(b0 + r) * T + t) * D,
                          gbytes, bar);
    };
    const int nchunks = b_end > b_begin ? (b_end - b_begin + CH - 1) / CH : 0;
    if (threadIdx.x == 0 && nchunks > 0) issue(0, 0);
    for (int i = 0; i < nchunks; ++i) {
        const int buf = i & 1;
        if (threadIdx.x == 0 && i + 1 < nchunks) issue(i + 1, buf ^ 1);   // its buffer was released by the last sync
        const bool ok = mbar_wait_bounded(smem_u32(&bars[buf]), (uint32_t)(i >> 1) & 1u, &s_abort, err, timeout_ns);
        if (__syncthreads_or(!ok)) {           // every thread leaves together; the copies in flight land first
            if (threadIdx.x == 0) {
                drain_copies(smem_u32(&bars[buf]), (uint32_t)(i >> 1) & 1u, timeout_ns);
                if (i + 1 < nchunks) drain_copies(smem_u32(&bars[buf ^ 1]), (uint32_t)((i + 1) >> 1) & 1u, timeout_ns);
            }
            break;
        }
        const int b0 = b_begin + i * CH;
        const int nrows = min(CH, b_end - b0);
        const Tz* zs = zbuf + (size_t)buf * CH * D;
        const float* gs = gbuf + (size_t)buf * CH * D;
        if (warp < nrows) {
            const Tz* z = zs + (size_t)warp * D;
            const float* gr = gs + (size_t)warp * D;
            const float shift = to_f32(z[0]);
            float s1 = 0.f, s2 = 0.f, sq = 0.f, sqz = 0.f;
            for (int k = 4 * lane; k < D; k += 128) {
                const float4 zz = ld4_any<Tz>(z + k);
                const float4 gg = *reinterpret_cast<const float4*>(gr + k);
                const float4 ga = __ldg(reinterpret_cast<const float4*>(g2 + k));
                const float d0 = zz.x - shift, d1 = zz.y - shift, d2 = zz.z - shift, d3 = zz.w - shift;
                const float q0 = gg.x * ga.x, q1 = gg.y * ga.y, q2 = gg.z * ga.z, q3 = gg.w * ga.w;
                s1 += (d0 + d1) + (d2 + d3);
                s2 = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, s2))));
                sq += (q0 + q1) + (q2 + q3);
                sqz = fmaf(q0, d0, fmaf(q1, d1, fmaf(q2, d2, fmaf(q3, d3, sqz))));
            }
            s1 = warp_sum(s1);
            s2 = warp_sum(s2);
            sq = warp_sum(sq);
            sqz = warp_sum(sqz);
            const float dm = s1 / (float)D;
            const float rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
            if (lane == 0)
                st[warp] = make_float4(shift + dm, rstd, sq / (float)D, rstd * (sqz - dm * sq) / (float)D);
        }
        __syncthreads();
        for (int r = 0; r < nrows; ++r) {
            const float4 s = st[r];
            float* dz = dZ + ((size_t)t * Bcap + b0 + r) * D;
#pragma unroll
            for (int j = 0; j < kLn2MaxPairs; ++j) {
                const int pidx = threadIdx.x + j * kLn2Threads;
                if (pidx < npairs) {
                    const int k = 2 * pidx;
                    const float2 zz = ld2_any<Tz>(zs + (size_t)r * D + k);
                    const float2 gk = *reinterpret_cast<const float2*>(gs + (size_t)r * D + k);
                    const float2 ga = __ldg(reinterpret_cast<const float2*>(g2 + k));
                    const float zh0 = (zz.x - s.x) * s.y, zh1 = (zz.y - s.x) * s.y;
                    float2 d;
                    d.x = (gk.x * ga.x - s.z - zh0 * s.w) * s.y;
                    d.y = (gk.y * ga.y - s.z - zh1 * s.w) * s.y;
                    *reinterpret_cast<float2*>(dz + k) = d;
                    amax = fmaxf(amax, fmaxf(fabsf(d.x), fabsf(d.y)));
                    adb[j].x += d.x;
                    adb[j].y += d.y;
                    adg[j].x = fmaf(gk.x, zh0, adg[j].x);
                    adg[j].y = fmaf(gk.y, zh1, adg[j].y);
                    adbe[j].x += gk.x;
                    adbe[j].y += gk.y;
                }
            }
        }
        __syncthreads();                       // buffer `buf` is free for chunk i + 2
    }
    const size_t prow = ((size_t)t * nbx + bx) * D;
#pragma unroll
    for (int j = 0; j < kLn2MaxPairs; ++j) {
        const int pidx = threadIdx.x + j * kLn2Threads;
        if (pidx < npairs) {
            *reinterpret_cast<float2*>(part_db2 + prow + 2 * pidx) = adb[j];
            *reinterpret_cast<float2*>(part_dg2 + prow + 2 * pidx) = adg[j];
            *reinterpret_cast<float2*>(part_dbe2 + prow + 2 * pidx) = adbe[j];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < kLn2Threads / 32; ++w) m = fmaxf(m, wmax[w]);
        part_max[(size_t)t * nbx + bx] = m;
    }
}

// ---- per-token scale of the gradient operands ----------------------------------------
// s_t = 2^(9 - e) where m = f 2^e, f in [0.5, 1), is token t's largest |dZ|, so
// s_t m lies in [2^8, 2^9): fp16 keeps 11 significant bits for every value down
// to 2^-14 / s_t and has 2^7 of headroom above for dU.  Powers of two make the
// scaling and its undoing exact.
__global__ void grad_scale_kernel(const float* __restrict__ dZ, const float* __restrict__ part_max, int nblk,
                                  float* __restrict__ inv_scale, __half* __restrict__ dZh, int B, int D, int Bcap) {
    __shared__ float sc;
    const int t = blockIdx.y;
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int i = 0; i < nblk; ++i) m = fmaxf(m, part_max[(size_t)t * nblk + i]);
        float s = 1.0f;
        if (m > 0.f && m <= 3.0e38f) {
            int e;
            frexpf(m, &e);
            s = ldexpf(1.0f, 9 - e);
        }
        sc = s;
        if (blockIdx.x == 0) inv_scale[t] = 1.0f / s;
    }
    __syncthreads();
    const float s = sc;
    const long long n = (long long)B * D;
    const float* src = dZ + (size_t)t * Bcap * D;
    __half* dst = dZh + (size_t)t * Bcap * D;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        dst[i] = __float2half_rn(sat_f16(src[i] * s));
}

__global__ void bf16_to_f16_kernel(const __nv_bfloat16* __restrict__ in, __half* __restrict__ out, long long n) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        out[i] = __float2half_rn(sat_f16(__bfloat162float(in[i])));
}

// ---- LN1 + mixing backward ---------------------------------------------------------
// One CTA per sample at a time (persistent over samples), from yhat and rstd
// of the LN1 recompute:
//   1. per row t (a warp): mean(q) and mean(q yhat), q = dS[t] gamma1;
//   2. per element (a thread per column k = c q + r, rows t in turn):
//        dX[t][k] = F(t, k) + F(c, t q + r),
//      F(u, j) = rstd_u (dS[u][j] gamma1[j] - mean(q)_u - yhat[u][j] mean(q yhat)_u),
//      i.e. dY + P^T dY with dY = F never stored: the transposed partner of
//      element (t, c q + r) is (c, t q + r).  A thread's columns (and so c
//      and r) are fixed, so no division runs per element.
// The thread owning column k also sums dS[t][k] yhat[t][k] and dS[t][k] over
// the rows of its samples (the CTA's dgamma1, dbeta1 partials).
template <typename Tyh>
__global__ void __launch_bounds__(kLn1Threads)
ln1_mix_backward_kernel(const Tyh* __restrict__ Yh, const float* __restrict__ rstdv, const float* __restrict__ dS,
                        const float* __restrict__ g1, float* __restrict__ dX, float* __restrict__ part_dg1,
                        float* __restrict__ part_dbe1, int B, int T, int D, int Bcap, QDiv qd) {
    __shared__ float4 st[kRowMaxT];                   // (rstd, mean(q), mean(q yhat)) per row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = (int)qd.q;
    int cc_[kLn1MaxCols], rr_[kLn1MaxCols];
#pragma unroll
    for (int j = 0; j < kLn1MaxCols; ++j) {
        const int k = threadIdx.x + j * kLn1Threads;
        cc_[j] = k < D ? qd.div(k) : 0;
        rr_[j] = k - cc_[j] * q;
    }
    float adg[kLn1MaxCols], adbe[kLn1MaxCols];
#pragma unroll
    for (int j = 0; j < kLn1MaxCols; ++j) adg[j] = adbe[j] = 0.f;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        __syncthreads();                              // the previous sample is done with st
        for (int t = warp; t < T; t += kLn1Threads / 32) {
            const size_t o = ((size_t)t * Bcap + b) * D;
            float mq = 0.f, mqy = 0.f;
            for (int k = lane; k < D; k += 32) {
                const float qk = dS[o + k] * g1[k];
                mq += qk;
                mqy = fmaf(qk, to_f32(Yh[o + k]), mqy);
            }
            mq = warp_sum(mq);
            mqy = warp_sum(mqy);
            if (lane == 0) st[t] = make_float4(rstdv[(size_t)t * Bcap + b], mq / (float)D, mqy / (float)D, 0.f);
        }
        __syncthreads();
        float* out = dX + (size_t)b * T * D;
        for (int t = 0; t < T; ++t) {
            const float4 s1 = st[t];
            const size_t o1 = ((size_t)t * Bcap + b) * D;
#pragma unroll
            for (int j = 0; j < kLn1MaxCols; ++j) {
                const int k = threadIdx.x + j * kLn1Threads;
                if (k < D) {
                    const int c = cc_[j];
                    const int k2 = t * q + rr_[j];            // the partner element (c, t q + r)
                    const float4 s2 = st[c];
                    const size_t o2 = ((size_t)c * Bcap + b) * D + k2;
                    const float yh1 = to_f32(Yh[o1 + k]);
                    const float yh2 = to_f32(Yh[o2]);
                    const float d1 = dS[o1 + k];
                    const float d2 = dS[o2];
                    const float f1 = (d1 * g1[k] - s1.y - yh1 * s1.z) * s1.x;
                    const float f2 = (d2 * g1[k2] - s2.y - yh2 * s2.z) * s2.x;
                    out[(size_t)t * D + k] = f1 + f2;
                    adg[j] = fmaf(d1, yh1, adg[j]);
                    adbe[j] += d1;
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kLn1MaxCols; ++j) {
        const int k = threadIdx.x + j * kLn1Threads;
        if (k < D) {
            part_dg1[(size_t)blockIdx.x * D + k] = adg[j];
            part_dbe1[(size_t)blockIdx.x * D + k] = adbe[j];
        }
    }
}

// The same with two adjacent columns per thread step (q and D even, D a
// multiple of 4): column pairs (k, k + 1) with k even have their partners at
// (c, t q + r) and (c, t q + r + 1), so every load and store moves a pair, and
// the row statistics read 4 columns per lane step.
template <typename Tyh>
struct Pair2;
template <>
struct Pair2<__half> {
    static __device__ __forceinline__ float2 ld(const __half* p) {
        return __half22float2(*reinterpret_cast<const __half2*>(p));
    }
    static __device__ __forceinline__ float4 ld4(const __half* p) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
};
template <>
struct Pair2<float> {
    static __device__ __forceinline__ float2 ld(const float* p) { return *reinterpret_cast<const float2*>(p); }
    static __device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
};

constexpr int kLn1MaxPairs = 3072 / 2 / kLn1Threads;

template <typename Tyh>
__global__ void __launch_bounds__(kLn1Threads, 3)
ln1_mix_backward_pair_kernel(const Tyh* __restrict__ Yh, const float* __restrict__ rstdv,
                             const float* __restrict__ dS, const float* __restrict__ g1, float* __restrict__ dX,
                             float* __restrict__ part_dg1, float* __restrict__ part_dbe1, int B, int T, int D, int Bcap,
                             QDiv qd) {
    __shared__ float4 st[kRowMaxT];                   // (rstd, mean(q), mean(q yhat)) per row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = (int)qd.q;
    const int npairs = D / 2;
    int cc_[kLn1MaxPairs], rr_[kLn1MaxPairs];
#pragma unroll
    for (int j = 0; j < kLn1MaxPairs; ++j) {
        const int k = 2 * (threadIdx.x + j * kLn1Threads);
        cc_[j] = k < D ? qd.div(k) : 0;
        rr_[j] = k - cc_[j] * q;
    }
    float2 adg[kLn1MaxPairs], adbe[kLn1MaxPairs];
#pragma unroll
    for (int j = 0; j < kLn1MaxPairs; ++j) adg[j] = adbe[j] = make_float2(0.f, 0.f);
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        __syncthreads();                              // the previous sample is done with st
        for (int t = warp; t < T; t += kLn1Threads / 32) {
            const size_t o = ((size_t)t * Bcap + b) * D;
            float mq = 0.f, mqy = 0.f;
            for (int k = 4 * lane; k < D; k += 128) {
                const float4 d = *reinterpret_cast<const float4*>(dS + o + k);
                const float4 gg = *reinterpret_cast<const float4*>(g1 + k);
                const float4 y = Pair2<Tyh>::ld4(Yh + o + k);
                const float q0 = d.x * gg.x, q1 = d.y * gg.y, q2 = d.z * gg.z, q3 = d.w * gg.w;
                mq += (q0 + q1) + (q2 + q3);
                mqy = fmaf(q0, y.x, fmaf(q1, y.y, fmaf(q2, y.z, fmaf(q3, y.w, mqy))));
            }
            mq = warp_sum(mq);
            mqy = warp_sum(mqy);
            if (lane == 0) st[t] = make_float4(rstdv[(size_t)t * Bcap + b], mq / (float)D, mqy / (float)D, 0.f);
        }
        __syncthreads();
        float* out = dX + (size_t)b * T * D;
#pragma unroll 4
        for (int t = 0; t < T; ++t) {
            const float4 s1 = st[t];
            const size_t o1 = ((size_t)t * Bcap + b) * D;
#pragma unroll
            for (int j = 0; j < kLn1MaxPairs; ++j) {
                const int pidx = threadIdx.x + j * kLn1Threads;
                if (pidx < npairs) {
                    const int k = 2 * pidx;
                    const int c = cc_[j];
                    const int k2 = t * q + rr_[j];            // partners (c, k2) and (c, k2 + 1)
                    const float4 s2 = st[c];
                    const size_t o2 = ((size_t)c * Bcap + b) * D + k2;
                    const float2 y1 = Pair2<Tyh>::ld(Yh + o1 + k);
                    const float2 y2 = Pair2<Tyh>::ld(Yh + o2);
                    const float2 d1 = *reinterpret_cast<const float2*>(dS + o1 + k);
                    const float2 d2 = *reinterpret_cast<const float2*>(dS + o2);
                    const float2 ga = *reinterpret_cast<const float2*>(g1 + k);
                    const float2 gb = *reinterpret_cast<const float2*>(g1 + k2);
                    float2 r;
                    r.x = (d1.x * ga.x - s1.y - y1.x * s1.z) * s1.x + (d2.x * gb.x - s2.y - y2.x * s2.z) * s2.x;
                    r.y = (d1.y * ga.y - s1.y - y1.y * s1.z) * s1.x + (d2.y * gb.y - s2.y - y2.y * s2.z) * s2.x;
                    *reinterpret_cast<float2*>(out + (size_t)t * D + k) = r;
                    adg[j].x = fmaf(d1.x, y1.x, adg[j].x);
                    adg[j].y = fmaf(d1.y, y1.y, adg[j].y);
                    adbe[j].x += d1.x;
                    adbe[j].y += d1.y;
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kLn1MaxPairs; ++j) {
        const int pidx = threadIdx.x + j * kLn1Threads;
        if (pidx < npairs) {
            *reinterpret_cast<float2*>(part_dg1 + (size_t)blockIdx.x * D + 2 * pidx) = adg[j];
            *reinterpret_cast<float2*>(part_dbe1 + (size_t)blockIdx.x * D + 2 * pidx) = adbe[j];
        }
    }
}

// Staged variant (T D floats fit in shared memory, q even, D a multiple of 4):
// one 1024-thread CTA per SM walks the samples; a sample's dS rows arrive in
// shared memory by bulk copies (one per token row, completion counted on an
// mbarrier with a bounded wait), so dS is read from HBM once and both the
// row statistics and the transposed partners read it from shared memory.
// yhat stays in global memory: with one sample per SM in flight its rows stay
// in L2 between the two phases.
constexpr int kLn1StThreads = 1024;
constexpr int kLn1StMaxPairs = 3072 / 2 / kLn1StThreads + 1;

template <typename Tyh>
__global__ void __launch_bounds__(kLn1StThreads, 1)
ln1_mix_backward_staged_kernel(const Tyh* __restrict__ Yh, const float* __restrict__ rstdv,
                               const float* __restrict__ dS, const float* __restrict__ g1, float* __restrict__ dX,
                               float* __restrict__ part_dg1, float* __restrict__ part_dbe1, int B, int T, int D,
                               int Bcap, QDiv qd, int* err, unsigned long long timeout_ns) {
    extern __shared__ float4 smem4[];
    float4* st = smem4;                                      // [T] (rstd, mean(q), mean(q yhat))
    float* ds = reinterpret_cast<float*>(smem4 + T);         // [T][D] the sample's dS rows
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = (int)qd.q;
    const int npairs = D / 2;
    int cc_[kLn1StMaxPairs], rr_[kLn1StMaxPairs];
#pragma unroll
    for (int j = 0; j < kLn1StMaxPairs; ++j) {
        const int k = 2 * (threadIdx.x + j * kLn1StThreads);
        cc_[j] = k < D ? qd.div(k) : 0;
        rr_[j] = k - cc_[j] * q;
    }
    float2 adg[kLn1StMaxPairs], adbe[kLn1StMaxPairs];
#pragma unroll
    for (int j = 0; j < kLn1StMaxPairs; ++j) adg[j] = adbe[j] = make_float2(0.f, 0.f);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t row_bytes = (uint32_t)D * 4u;
    uint32_t phase = 0;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        __syncthreads();                                     // the previous sample is done with ds and st
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();                        // generic reads of ds before the async writes
            mbar_arrive_expect_tx(smem_u32(&bar), row_bytes * (uint32_t)T);
            for (int t = 0; t < T; ++t)
                bulk_copy_g2s(smem_u32(ds + (size_t)t * D), dS + ((size_t)t * Bcap + b) * D, row_bytes,
                              smem_u32(&bar));
        }
        const bool ok = mbar_wait_bounded(smem_u32(&bar), phase, &s_abort, err, timeout_ns);
        if (__syncthreads_or(!ok)) {                         // every thread leaves together on a timeout
            if (threadIdx.x == 0) drain_copies(smem_u32(&bar), phase, timeout_ns);
            break;
        }
        phase ^= 1u;
        for (int t = warp; t < T; t += kLn1StThreads / 32) {
            const size_t o = ((size_t)t * Bcap + b) * D;
            const float* dr = ds + (size_t)t * D;
            float mq = 0.f, mqy = 0.f;
            for (int k = 4 * lane; k < D; k += 128) {
                const float4 d = *reinterpret_cast<const float4*>(dr + k);
                const float4 gg = __ldg(reinterpret_cast<const float4*>(g1 + k));
                const float4 y = Pair2<Tyh>::ld4(Yh + o + k);
                const float q0 = d.x * gg.x, q1 = d.y * gg.y, q2 = d.z * gg.z, q3 = d.w * gg.w;
                mq += (q0 + q1) + (q2 + q3);
                mqy = fmaf(q0, y.x, fmaf(q1, y.y, fmaf(q2, y.z, fmaf(q3, y.w, mqy))));
            }
            mq = warp_sum(mq);
            mqy = warp_sum(mqy);
            if (lane == 0) st[t] = make_float4(rstdv[(size_t)t * Bcap + b], mq / (float)D, mqy / (float)D, 0.f);
        }
        __syncthreads();
        float* out = dX + (size_t)b * T * D;
#pragma unroll
        for (int j = 0; j < kLn1StMaxPairs; ++j) {
            const int pidx = threadIdx.x + j * kLn1StThreads;
            if (pidx < npairs) {
                const int k = 2 * pidx;
                const int c = cc_[j];
                const float4 s2 = st[c];
                const float2 ga = __ldg(reinterpret_cast<const float2*>(g1 + k));
                for (int t = 0; t < T; ++t) {
                    const float4 s1 = st[t];
                    const int k2 = t * q + rr_[j];           // partners (c, k2) and (c, k2 + 1)
                    const float2 gb = __ldg(reinterpret_cast<const float2*>(g1 + k2));
                    const float2 y1 = Pair2<Tyh>::ld(Yh + ((size_t)t * Bcap + b) * D + k);
                    const float2 y2 = Pair2<Tyh>::ld(Yh + ((size_t)c * Bcap + b) * D + k2);
                    const float2 d1 = *reinterpret_cast<const float2*>(ds + (size_t)t * D + k);
                    const float2 d2 = *reinterpret_cast<const float2*>(ds + (size_t)c * D + k2);
                    float2 r;
                    r.x = (d1.x * ga.x - s1.y - y1.x * s1.z) * s1.x + (d2.x * gb.x - s2.y - y2.x * s2.z) * s2.x;
                    r.y = (d1.y * ga.y - s1.y - y1.y * s1.z) * s1.x + (d2.y * gb.y - s2.y - y2.y * s2.z) * s2.x;
                    *reinterpret_cast<float2*>(out + (size_t)t * D + k) = r;
                    adg[j].x = fmaf(d1.x, y1.x, adg[j].x);
                    adg[j].y = fmaf(d1.y, y1.y, adg[j].y);
                    adbe[j].x += d1.x;
                    adbe[j].y += d1.y;
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kLn1StMaxPairs; ++j) {
        const int pidx = threadIdx.x + j * kLn1StThreads;
        if (pidx < npairs) {
            *reinterpret_cast<float2*>(part_dg1 + (size_t)blockIdx.x * D + 2 * pidx) = adg[j];
            *reinterpret_cast<float2*>(part_dbe1 + (size_t)blockIdx.x * D + 2 * pidx) = adbe[j];
        }
    }
}

// ---- reductions ------------------------------------------------------------------
__global__ void sum_rows_kernel(const float* __restrict__ in, float* __restrict__ out, int R, int N) {
    const int g = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const float* p = in + (size_t)g * R * N + n;
    float s = 0.f;
    for (int r = 0; r < R; ++r) s += p[(size_t)r * N];
    out[(size_t)g * N + n] = s;
}

__global__ void sum_groups_kernel(const float* __restrict__ in, float* __restrict__ out, int G, int N) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += in[(size_t)g * N + n];
    out[n] = s;
}

// G[b][t][k] = dP[b][k] / T: a thread per (sample, 4 columns) writes its float4 to every token row.
__global__ void pool_backward_kernel(const float* __restrict__ dP, float* __restrict__ G, int B, int T, int D) {
    const int d4 = D / 4;
    const long long n = (long long)B * d4;
    const float inv = 1.0f / (float)T;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(i / d4), j = (int)(i - (long long)b * d4);
        float4 v = reinterpret_cast<const float4*>(dP + (size_t)b * D)[j];
        v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
        float4* o = reinterpret_cast<float4*>(G + (size_t)b * T * D) + j;
        for (int t = 0; t < T; ++t) o[(size_t)t * d4] = v;
    }
}

// The same for D not a multiple of 4.
__global__ void pool_backward_scalar_kernel(const float* __restrict__ dP, float* __restrict__ G, int B, int T, int D) {
    const long long n = (long long)B * D;
    const float inv = 1.0f / (float)T;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(i / D), k = (int)(i - (long long)b * D);
        const float v = dP[i] * inv;
        for (int t = 0; t < T; ++t) G[((size_t)b * T + t) * D + k] = v;
    }
}

__global__ void debug_gelu_grad_kernel(const float* __restrict__ u, float* __restrict__ out, long long n) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const GeluPair p = gelu_with_grad(u[i]);
        out[2 * i] = p.value;
        out[2 * i + 1] = p.grad;
    }
}

int grid_for(long long n, int threads, int cap) {
    long long g = (n + threads - 1) / threads;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}


}  // namespace

cudaError_t launch_ln1_recompute(Act act, bool x_f32, const void* X, void* S, void* Yh, float* rstd, const float* g1,
                                 const float* be1, int B, int T, int D, int Bcap, float eps, int num_sms,
                                 cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T, 8, num_sms * 8);
    const QDiv qd = make_qdiv(D / T);
    const size_t esz = (act == Act::F32 || x_f32) ? 4 : 2;
    const size_t smem = (size_t)T * D * esz;
    if ((D / T) % 2 == 0 && smem % 16 == 0 && smem <= kLn1RecSmemLimit && act != Act::F32) {
        // two CTAs of 512 threads per SM when two samples fit (bf16 inputs at the
        // 1B width), else one of 1024 (float32 inputs)
        const int per_sm = smem <= 100 * 1024 ? 2 : 1;
        const int threads = per_sm == 2 ? kLn1RecThreads / 2 : kLn1RecThreads;
        const int sgrid = B < num_sms * per_sm ? B : num_sms * per_sm;
        if (x_f32) {
            auto k = ln1_recompute_staged_kernel<float, __half, __half>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            k<<<sgrid, threads, smem, s>>>((const float*)X, (__half*)S, (__half*)Yh, rstd, g1, be1, B, T, D, Bcap,
                                            eps, qd);
        } else {
            auto k = ln1_recompute_staged_kernel<__nv_bfloat16, __half, __half>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            k<<<sgrid, threads, smem, s>>>((const __nv_bfloat16*)X, (__half*)S, (__half*)Yh, rstd, g1, be1, B, T, D,
                                            Bcap, eps, qd);
        }
        return cudaGetLastError();
    }
    if ((D / T) % 2 == 0) {
        if (act == Act::F32)
            ln1_recompute_pair_kernel<float, float, float><<<grid, 256, 0, s>>>(
                (const float*)X, (float*)S, (float*)Yh, rstd, g1, be1, B, T, D, Bcap, eps, qd);
        else if (x_f32)
            ln1_recompute_pair_kernel<float, __half, __half><<<grid, 256, 0, s>>>(
                (const float*)X, (__half*)S, (__half*)Yh, rstd, g1, be1, B, T, D, Bcap, eps, qd);
        else
            ln1_recompute_pair_kernel<__nv_bfloat16, __half, __half><<<grid, 256, 0, s>>>(
                (const __nv_bfloat16*)X, (__half*)S, (__half*)Yh, rstd, g1, be1, B, T, D, Bcap, eps, qd);
        return cudaGetLastError();
    }
    if (act == Act::F32)
        ln1_recompute_kernel<float, float, float><<<grid, 256, 0, s>>>((const float*)X, (float*)S, (float*)Yh, rstd,
                                                                        g1, be1, B, T, D, Bcap, eps, qd);
    else if (x_f32)
        ln1_recompute_kernel<float, __half, __half><<<grid, 256, 0, s>>>((const float*)X, (__half*)S, (__half*)Yh,
                                                                          rstd, g1, be1, B, T, D, Bcap, eps, qd);
    else
        ln1_recompute_kernel<__nv_bfloat16, __half, __half><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16*)X, (__half*)S, (__half*)Yh, rstd, g1, be1, B, T, D, Bcap, eps, qd);
    return cudaGetLastError();
}

constexpr int kLn2DbSmemLimit = 220 * 1024;
constexpr int kLn2DbChunk = 4;             // rows per chunk of the double-buffered kernel

size_t ln2_db_bytes(Act act, int D) {
    const size_t zsz = act == Act::F32 ? 4 : 2;
    return kLn2DbChunk * sizeof(float4) + 2 * (size_t)kLn2DbChunk * D * (4 + zsz);
}

bool ln2_bwd_double_buffered(Act act, int D) {
    return D % 8 == 0 && ln2_db_bytes(act, D) <= (size_t)kLn2DbSmemLimit;
}

// CTAs per token: as many as fill the SMs in one wave (rounded down, so that
// no CTA waits for a second wave), at most one per chunk.
int ln2_bwd_blocks(Act act, int B, int T, int D, int num_sms) {
    int per_sm = 3;
    int chunk = kLn2Chunk;
    if (ln2_bwd_double_buffered(act, D)) {
        per_sm = (int)((227 * 1024) / (ln2_db_bytes(act, D) + 1024));
        if (per_sm > 3) per_sm = 3;
        if (per_sm < 1) per_sm = 1;
        chunk = kLn2DbChunk;
    }
    const int want = per_sm * num_sms / T;
    const int most = (B + chunk - 1) / chunk;
    const int n = want < most ? want : most;
    return n < 1 ? 1 : n;
}

cudaError_t launch_ln2_backward(Act act, const void* Z, const float* G, const float* g2, float* dZ, float* part_db2,
                                float* part_dg2, float* part_dbe2, float* part_max, int B, int T, int D, int Bcap,
                                float eps, int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (D > kLn2MaxCols * kLn2Threads) return cudaErrorNotSupported;
    const int nbx = ln2_bwd_blocks(act, B, T, D, num_sms);
    const dim3 grid(nbx, T);
    const size_t zsz = act == Act::F32 ? 4 : 2;
    if (ln2_bwd_double_buffered(act, D)) {
        const int per = ((B + nbx - 1) / nbx + kLn2DbChunk - 1) / kLn2DbChunk * kLn2DbChunk;
        const size_t dbytes = ln2_db_bytes(act, D);
        if (act == Act::F32) {
            auto k = ln2_backward_db_kernel<float, kLn2DbChunk>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dbytes);
            if (e != cudaSuccess) return e;
            k<<<grid, kLn2Threads, dbytes, s>>>((const float*)Z, G, g2, dZ, part_db2, part_dg2, part_dbe2, part_max,
                                                B, T, D, Bcap, eps, per, err, timeout_ns);
        } else {
            auto k = ln2_backward_db_kernel<__half, kLn2DbChunk>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dbytes);
            if (e != cudaSuccess) return e;
            k<<<grid, kLn2Threads, dbytes, s>>>((const __half*)Z, G, g2, dZ, part_db2, part_dg2, part_dbe2, part_max,
                                                B, T, D, Bcap, eps, per, err, timeout_ns);
        }
        return cudaGetLastError();
    }
    const int per = ((B + nbx - 1) / nbx + kLn2Chunk - 1) / kLn2Chunk * kLn2Chunk;
    const size_t bytes = kLn2Chunk * sizeof(float4) + (size_t)kLn2Chunk * D * (4 + zsz);
    const bool vec = D % 8 == 0;               // whole 16-byte lines of fp16 rows and float4 of float rows
    if (vec) {
        if (act == Act::F32) {
            auto k = ln2_backward_vec_kernel<float>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e != cudaSuccess) return e;
            k<<<grid, kLn2Threads, bytes, s>>>((const float*)Z, G, g2, dZ, part_db2, part_dg2, part_dbe2, part_max,
                                               B, T, D, Bcap, eps, per);
        } else {
            auto k = ln2_backward_vec_kernel<__half>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e != cudaSuccess) return e;
            k<<<grid, kLn2Threads, bytes, s>>>((const __half*)Z, G, g2, dZ, part_db2, part_dg2, part_dbe2, part_max,
                                               B, T, D, Bcap, eps, per);
        }
        return cudaGetLastError();
    }
    if (act == Act::F32) {
        auto k = ln2_backward_kernel<float>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        k<<<grid, kLn2Threads, bytes, s>>>((const float*)Z, G, g2, dZ, part_db2, part_dg2, part_dbe2, part_max, B, T,
                                           D, Bcap, eps, per);
    } else {
        auto k = ln2_backward_kernel<__half>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        k<<<grid, kLn2Threads, bytes, s>>>((const __half*)Z, G, g2, dZ, part_db2, part_dg2, part_dbe2, part_max, B,
                                           T, D, Bcap, eps, per);
    }
    return cudaGetLastError();
}

cudaError_t launch_grad_scale(const float* dZ, const float* part_max, int nblk, float* inv_scale, void* dZh, int B,
                              int T, int D, int Bcap, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const dim3 grid((unsigned)grid_for((long long)B * D, 256, 64), T);
    grad_scale_kernel<<<grid, 256, 0, s>>>(dZ, part_max, nblk, inv_scale, (__half*)dZh, B, D, Bcap);
    return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(const void* in, void* out, long long n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    bf16_to_f16_kernel<<<grid_for(n, 256, 8192), 256, 0, s>>>((const __nv_bfloat16*)in, (__half*)out, n);
    return cudaGetLastError();
}

constexpr int kLn1StagedSmemLimit = 220 * 1024;
bool ln1_bwd_staged(int T, int D);

int ln1_bwd_grid(int B, int T, int D, int num_sms) {
    const int cap = ln1_bwd_staged(T, D) ? num_sms : num_sms * 4;
    return B < cap ? (B < 1 ? 1 : B) : cap;
}

bool ln1_bwd_staged(int T, int D) {
    return (D / T) % 2 == 0 && D % 4 == 0 &&
           (size_t)T * sizeof(float4) + (size_t)T * D * sizeof(float) <= (size_t)kLn1StagedSmemLimit;
}

cudaError_t launch_ln1_mix_backward(Act act, const void* Yh, const float* rstd, const float* dS, const float* g1,
                                    float* dX, float* part_dg1, float* part_dbe1, int B, int T, int D, int Bcap,
                                    int grid, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (D > kLn1MaxCols * kLn1Threads || T > kRowMaxT) return cudaErrorNotSupported;
    const QDiv qd = make_qdiv(D / T);
    if (ln1_bwd_staged(T, D)) {
        const size_t bytes = (size_t)T * sizeof(float4) + (size_t)T * D * sizeof(float);
        if (act == Act::F32) {
            auto k = ln1_mix_backward_staged_kernel<float>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e != cudaSuccess) return e;
            k<<<grid, kLn1StThreads, bytes, s>>>((const float*)Yh, rstd, dS, g1, dX, part_dg1, part_dbe1, B, T, D,
                                                 Bcap, qd, err, timeout_ns);
        } else {
            auto k = ln1_mix_backward_staged_kernel<__half>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e != cudaSuccess) return e;
            k<<<grid, kLn1StThreads, bytes, s>>>((const __half*)Yh, rstd, dS, g1, dX, part_dg1, part_dbe1, B, T, D,
                                                 Bcap, qd, err, timeout_ns);
        }
        return cudaGetLastError();
    }
    const bool pairs = (D / T) % 2 == 0 && D % 4 == 0;
    if (act == Act::F32) {
        if (pairs)
            ln1_mix_backward_pair_kernel<float><<<grid, kLn1Threads, 0, s>>>((const float*)Yh, rstd, dS, g1, dX,
                                                                             part_dg1, part_dbe1, B, T, D, Bcap, qd);
        else
            ln1_mix_backward_kernel<float><<<grid, kLn1Threads, 0, s>>>((const float*)Yh, rstd, dS, g1, dX, part_dg1,
                                                                        part_dbe1, B, T, D, Bcap, qd);
    } else {
        if (pairs)
            ln1_mix_backward_pair_kernel<__half><<<grid, kLn1Threads, 0, s>>>((const __half*)Yh, rstd, dS, g1, dX,
                                                                              part_dg1, part_dbe1, B, T, D, Bcap, qd);
        else
            ln1_mix_backward_kernel<__half><<<grid, kLn1Threads, 0, s>>>((const __half*)Yh, rstd, dS, g1, dX,
                                                                         part_dg1, part_dbe1, B, T, D, Bcap, qd);
    }
    return cudaGetLastError();
}

cudaError_t launch_sum_rows(const float* in, float* out, float* out_all, int G, int R, int N, cudaStream_t s) {
    if (G <= 0 || N <= 0) return cudaSuccess;
    sum_rows_kernel<<<dim3((N + 255) / 256, G), 256, 0, s>>>(in, out, R, N);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || out_all == nullptr) return e;
    sum_groups_kernel<<<(N + 255) / 256, 256, 0, s>>>(out, out_all, G, N);
    return cudaGetLastError();
}

cudaError_t launch_pool_backward(const float* dpooled, float* G, int B, int T, int D, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const bool vec = D % 4 == 0 && (reinterpret_cast<uintptr_t>(dpooled) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
    if (vec)
        pool_backward_kernel<<<grid_for((long long)B * (D / 4), 256, 4096), 256, 0, s>>>(dpooled, G, B, T, D);
    else
        pool_backward_scalar_kernel<<<grid_for((long long)B * D, 256, 4096), 256, 0, s>>>(dpooled, G, B, T, D);
    return cudaGetLastError();
}

cudaError_t launch_debug_gelu_grad(const float* u, float* out, long long n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    debug_gelu_grad_kernel<<<grid_for(n, 256, 4096), 256, 0, s>>>(u, out, n);
    return cudaGetLastError();
}

}  // namespace rm
