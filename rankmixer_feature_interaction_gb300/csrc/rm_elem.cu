// Memory-bound kernels of the RankMixer block: TokenMixing fused with the
// first residual and LayerNorm, the second LayerNorm's finalisation (into the
// next layer's mixing, into a [B][T][D] output, or into mean pooling), and
// the small layout/packing kernels used at context creation.
//
// "RankMixer: Scaling Up Ranking Models in Industrial Recommenders", section
// 3.1 Eq. 1 and section 3.3.1 Eq. 3-5; "RankMixer 详解（1）" section 3.1 (the
// element map of the mixing) and section 3.3 (LayerNorm).
#include "rm_common.cuh"
#include "rm_internal.h"

namespace rm {
namespace {

constexpr int kMixThreads = 256;
constexpr int kMixWarps = kMixThreads / 32;

// LN affine applied to a finalised row element.  Every kernel that finalises
// LN2 (the next layer's mixing, the block output, the pool) uses this exact
// expression, so they all see the same float32 value of X_n.
__device__ __forceinline__ float ln_apply(float z, float mean, float rstd, float g, float b) {
    const float n = (z - mean) * rstd;
    return fmaf(n, g, b);
}

template <typename Tact> struct Vec2;
template <> struct Vec2<float> {
    using type = float2;
    __device__ static float2 load(const float* p) { return *reinterpret_cast<const float2*>(p); }
    __device__ static void store(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
    __device__ static void split(float2 v, float& a, float& b) { a = v.x; b = v.y; }
};
template <> struct Vec2<__half> {
    __device__ static __half2 load(const __half* p) { return *reinterpret_cast<const __half2*>(p); }
    __device__ static void store(__half* p, float a, float b) {
        *reinterpret_cast<__half2*>(p) = __floats2half2_rn(sat_f16(a), sat_f16(b));
    }
    __device__ static void split(__half2 v, float& a, float& b) {
        a = __low2float(v);
        b = __high2float(v);
    }
};
template <> struct Vec2<__nv_bfloat16> {
    __device__ static __nv_bfloat162 load(const __nv_bfloat16* p) {
        return *reinterpret_cast<const __nv_bfloat162*>(p);
    }
    __device__ static void store(__nv_bfloat16* p, float a, float b) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
    }
    __device__ static void split(__nv_bfloat162 v, float& a, float& b) {
        a = __low2float(v);
        b = __high2float(v);
    }
};

// ---------------------------------------------------------------------------
// Fused TokenMixing + residual + LN1.
// One CTA per sample (grid-stride), one warp per output row h:
//   y[j] = X[t][h q + r] + X[h][j],  j = t q + r          (mix + residual)
// with X read straight from global memory -- either the caller's X, or the
// previous layer's pre-LN2 rows Z finalised on the fly in float32 (the row
// statistics of the sample's T rows are merged once into shared memory).
// y stays in registers; mean and biased variance come from two warp
// reductions; S = LN1(y) is written token-major in the operand type Top
// (fp16 for bf16 contexts, float for float32 contexts).
// VEC = 2: each lane owns column pairs (needs q even, D % 64 == 0);
// VEC = 1: single columns (any q).  NI bounds D / (32 VEC).
// ---------------------------------------------------------------------------
constexpr int kMaxT = 128;

template <typename Tin, bool FROM_Z>
struct RowSrc {
    const Tin* X;
    const float* Z;
    const float* g2;
    const float* be2;
    const float* mean;
    const float* rstd;
    size_t xrow_stride;   // elements between token rows of one sample
    size_t zrow_stride;
    __device__ __forceinline__ float load1(int t, int c) const {
        if (FROM_Z) return ln_apply(Z[t * zrow_stride + c], mean[t], rstd[t], g2[c], be2[c]);
        return to_f32(X[t * xrow_stride + c]);
    }
    __device__ __forceinline__ void load2(int t, int c, float& v0, float& v1) const {
        if (FROM_Z) {
            const float2 z = *reinterpret_cast<const float2*>(Z + t * zrow_stride + c);
            const float2 g = *reinterpret_cast<const float2*>(g2 + c);
            const float2 be = *reinterpret_cast<const float2*>(be2 + c);
            v0 = ln_apply(z.x, mean[t], rstd[t], g.x, be.x);
            v1 = ln_apply(z.y, mean[t], rstd[t], g.y, be.y);
        } else {
            Vec2<Tin>::split(Vec2<Tin>::load(X + t * xrow_stride + c), v0, v1);
        }
    }
};

template <typename Tin, typename Top, bool FROM_Z, int VEC, int NI>
__global__ void __launch_bounds__(kMixThreads)
mix_ln1_kernel(const MixLnArgs a) {
    __shared__ float s_mean[kMaxT], s_rstd[kMaxT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, D = a.D, q = a.q;
    Top* S = reinterpret_cast<Top*>(a.S);

    for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        RowSrc<Tin, FROM_Z> src;
        src.X = reinterpret_cast<const Tin*>(a.X) + (size_t)b * T * D;
        src.Z = a.Z + (size_t)b * D;
        src.g2 = a.g2;
        src.be2 = a.be2;
        src.mean = s_mean;
        src.rstd = s_rstd;
        src.xrow_stride = (size_t)D;
        src.zrow_stride = (size_t)a.Bcap * D;
        if (FROM_Z) {
            for (int t = warp; t < T; t += kMixWarps) {
                float mean, rstd;
                merge_row_stats(a.stats + ((size_t)t * a.Bcap + b) * a.nchunk, a.nchunk, a.cw, D, a.eps, lane,
                                mean, rstd);
                if (lane == 0) {
                    s_mean[t] = mean;
                    s_rstd[t] = rstd;
                }
            }
            __syncthreads();
        }
        for (int h = warp; h < T; h += kMixWarps) {
            float y[NI * VEC];
            float sum = 0.f;
            if (VEC == 2) {
                const int ni = D >> 6;
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    if (i < ni) {
                        const int j = (i << 6) + (lane << 1);
                        const int t = j / q;
                        const int r = j - t * q;
                        float m0, m1, x0, x1;
                        src.load2(t, h * q + r, m0, m1);
                        src.load2(h, j, x0, x1);
                        y[2 * i] = m0 + x0;
                        y[2 * i + 1] = m1 + x1;
                        sum += y[2 * i] + y[2 * i + 1];
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const int j = (i << 5) + lane;
                    if (j < D) {
                        const int t = j / q;
                        const int r = j - t * q;
                        y[i] = src.load1(t, h * q + r) + src.load1(h, j);
                        sum += y[i];
                    }
                }
            }
            const float mean = warp_sum(sum) / (float)D;
            float sq = 0.f;
            if (VEC == 2) {
                const int ni = D >> 6;
#pragma unroll
                for (int i = 0; i < NI; ++i)
                    if (i < ni) {
                        const float d0 = y[2 * i] - mean, d1 = y[2 * i + 1] - mean;
                        sq += d0 * d0 + d1 * d1;
                    }
            } else {
#pragma unroll
                for (int i = 0; i < NI; ++i)
                    if ((i << 5) + lane < D) {
                        const float d = y[i] - mean;
                        sq += d * d;
                    }
            }
            const float rstd = rsqrtf(warp_sum(sq) / (float)D + a.eps);
            const size_t srow = ((size_t)h * a.Bcap + b) * D;
            if (VEC == 2) {
                const int ni = D >> 6;
#pragma unroll
                for (int i = 0; i < NI; ++i)
                    if (i < ni) {
                        const int j = (i << 6) + (lane << 1);
                        const float2 g = *reinterpret_cast<const float2*>(a.g1 + j);
                        const float2 be = *reinterpret_cast<const float2*>(a.be1 + j);
                        const float v0 = ln_apply(y[2 * i], mean, rstd, g.x, be.x);
                        const float v1 = ln_apply(y[2 * i + 1], mean, rstd, g.y, be.y);
                        Vec2<Top>::store(S + srow + j, v0, v1);
                    }
            } else {
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const int j = (i << 5) + lane;
                    if (j < D) S[srow + j] = from_f32<Top>(ln_apply(y[i], mean, rstd, a.g1[j], a.be1[j]));
                }
            }
        }
        if (FROM_Z) __syncthreads();   // s_mean / s_rstd are rewritten for the next sample
    }
}

template <typename Tin, typename Top, bool FROM_Z, int VEC, int NI>
cudaError_t launch_mix_inst(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    int grid = num_sms * 8;
    if (grid > a.B) grid = a.B;
    mix_ln1_kernel<Tin, Top, FROM_Z, VEC, NI><<<grid, kMixThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Top, bool FROM_Z>
cudaError_t launch_mix_dispatch(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    const bool vec2 = (a.q % 2 == 0) && (a.D % 64 == 0);
    if (vec2) {
        const int ni = a.D / 64;
        if (ni <= 4) return launch_mix_inst<Tin, Top, FROM_Z, 2, 4>(a, num_sms, s);
        if (ni <= 12) return launch_mix_inst<Tin, Top, FROM_Z, 2, 12>(a, num_sms, s);
        if (ni <= 24) return launch_mix_inst<Tin, Top, FROM_Z, 2, 24>(a, num_sms, s);
        if (ni <= 48) return launch_mix_inst<Tin, Top, FROM_Z, 2, 48>(a, num_sms, s);
        return cudaErrorNotSupported;
    }
    const int ni = (a.D + 31) / 32;
    if (ni <= 8) return launch_mix_inst<Tin, Top, FROM_Z, 1, 8>(a, num_sms, s);
    if (ni <= 48) return launch_mix_inst<Tin, Top, FROM_Z, 1, 48>(a, num_sms, s);
    return cudaErrorNotSupported;
}

// ---------------------------------------------------------------------------
// LN2 finalisation into a sample-major output: one warp per (b, t) row.
// ---------------------------------------------------------------------------
template <typename Tact>
__global__ void ln2_out_kernel(const float* __restrict__ Z, const float2* __restrict__ stats,
                               const float* __restrict__ g2, const float* __restrict__ be2, Tact* __restrict__ X,
                               int B, int T, int D, int Bcap, int nchunk, int cw, float eps) {
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = wid; r < (long long)B * T; r += nw) {
        const int b = (int)(r / T), t = (int)(r % T);
        const size_t zr = (size_t)t * Bcap + b;
        float mean, rstd;
        merge_row_stats(stats + zr * nchunk, nchunk, cw, D, eps, lane, mean, rstd);
        const float* z = Z + zr * D;
        Tact* x = X + ((size_t)b * T + t) * D;
        for (int j = lane; j < D; j += 32) x[j] = from_f32<Tact>(ln_apply(z[j], mean, rstd, g2[j], be2[j]));
    }
}

// ---------------------------------------------------------------------------
// Last LN2 finalisation + mean pooling over tokens, one CTA per sample.  The
// mean is taken over the float32 LN2 outputs in token order; XL (optional)
// receives them rounded to the activation dtype.
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 256;
constexpr int kPoolMaxT = 128;

template <typename Tact>
__global__ void __launch_bounds__(kPoolThreads)
pool_kernel(const float* __restrict__ Z, const float2* __restrict__ stats, const float* __restrict__ g2,
            const float* __restrict__ be2, float* __restrict__ pooled, Tact* __restrict__ XL, int B, int T, int D,
            int Bcap, int nchunk, int cw, float eps) {
    __shared__ float s_mean[kPoolMaxT], s_rstd[kPoolMaxT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        for (int t = warp; t < T; t += kPoolThreads / 32) {
            float mean, rstd;
            merge_row_stats(stats + ((size_t)t * Bcap + b) * nchunk, nchunk, cw, D, eps, lane, mean, rstd);
            if (lane == 0) {
                s_mean[t] = mean;
                s_rstd[t] = rstd;
            }
        }
        __syncthreads();
        for (int j = threadIdx.x; j < D; j += kPoolThreads) {
            const float g = g2[j], be = be2[j];
            float acc = 0.f;
            for (int t = 0; t < T; ++t) {
                const float v = ln_apply(Z[((size_t)t * Bcap + b) * D + j], s_mean[t], s_rstd[t], g, be);
                if (XL) XL[((size_t)b * T + t) * D + j] = from_f32<Tact>(v);
                acc += v;
            }
            pooled[(size_t)b * D + j] = acc / (float)T;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Row statistics (mean, M2) of full Z rows, two passes, one warp per row.
// ---------------------------------------------------------------------------
__global__ void rowstats_kernel(const float* __restrict__ Z, float2* __restrict__ stats, int B, int T, int D,
                                int Bcap) {
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = wid; r < (long long)B * T; r += nw) {
        const int t = (int)(r / B), b = (int)(r % B);
        const size_t zr = (size_t)t * Bcap + b;
        const float* z = Z + zr * D;
        float s = 0.f;
        for (int j = lane; j < D; j += 32) s += z[j];
        const float mean = warp_sum(s) / (float)D;
        float m2 = 0.f;
        for (int j = lane; j < D; j += 32) {
            const float d = z[j] - mean;
            m2 += d * d;
        }
        m2 = warp_sum(m2);
        if (lane == 0) stats[zr] = make_float2(mean, m2);
    }
}

// ---------------------------------------------------------------------------
// Layout helpers
// ---------------------------------------------------------------------------
template <typename Top, typename Tout>
__global__ void token_to_sample_kernel(const Top* __restrict__ src, Tout* __restrict__ dst, int B, int T, int D,
                                       int Bcap) {
    const long long n = (long long)B * T * D;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(i % D);
        const long long bt = i / D;
        const int t = (int)(bt % T), b = (int)(bt / T);
        dst[i] = from_f32<Tout>(to_f32(src[((size_t)t * Bcap + b) * D + j]));
    }
}

// Standalone TokenMixing on element bits: Y[b][h][t q + r] = X[b][t][h q + r].
template <typename E>
__global__ void token_mix_kernel(const E* __restrict__ X, E* __restrict__ Y, int B, int T, int D, int H) {
    const int q = D / H;
    const long long TD = (long long)T * D;
    const long long n = (long long)B * TD;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long b = i / TD;
        const long long o = i - b * TD;          // offset inside Y[b], row-major [H][T q]
        const int h = (int)(o / ((long long)T * q));
        const int c = (int)(o - (long long)h * T * q);
        const int t = c / q, r = c - t * q;
        Y[i] = X[b * TD + (long long)t * D + (long long)h * q + r];
    }
}

// out[g][c][r] = convert(in[g][r][c]), 32x32 tiles through shared memory.
template <typename Ein, typename Eout>
__global__ void transpose_kernel(const Ein* __restrict__ in, Eout* __restrict__ out, int R, int C) {
    __shared__ float tile[32][33];
    const size_t g = blockIdx.z;
    const Ein* src = in + g * (size_t)R * C;
    Eout* dst = out + g * (size_t)R * C;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < R && c < C) tile[i][threadIdx.x] = to_f32(src[(size_t)r * C + c]);
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < R && c < C) dst[(size_t)c * R + r] = from_f32<Eout>(tile[threadIdx.x][i]);
    }
}

template <typename Tin>
__global__ void to_f32_kernel(const Tin* __restrict__ in, float* __restrict__ out, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        out[i] = to_f32(in[i]);
}

__global__ void debug_wait_kernel(const int* flag, int* err, unsigned long long timeout_ns) {
    if (threadIdx.x != 0) return;
    const uint64_t t0 = globaltimer_ns();
    while (*(volatile const int*)flag == 0) {
        if (globaltimer_ns() - t0 > timeout_ns) {
            latch_error(err, kDevErrTimeout);
            return;
        }
        __nanosleep(1000);
    }
}

inline int grid_for(long long n, int threads, int cap = 152 * 16) {
    long long g = (n + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

}  // namespace

cudaError_t launch_mix_ln1(Act act, bool from_z, const MixLnArgs& a, int num_sms, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (act == Act::BF16)
        return from_z ? launch_mix_dispatch<__nv_bfloat16, __half, true>(a, num_sms, s)
                      : launch_mix_dispatch<__nv_bfloat16, __half, false>(a, num_sms, s);
    return from_z ? launch_mix_dispatch<float, float, true>(a, num_sms, s)
                  : launch_mix_dispatch<float, float, false>(a, num_sms, s);
}

cudaError_t launch_ln2_out(Act act, const float* Z, const float2* stats, const float* g2, const float* be2,
                           void* X_out, int B, int T, int D, int Bcap, int nchunk, int cw, float eps, int num_sms,
                           cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T * 32, 256, num_sms * 8);
    if (act == Act::BF16)
        ln2_out_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(Z, stats, g2, be2, (__nv_bfloat16*)X_out, B, T, D, Bcap,
                                                            nchunk, cw, eps);
    else
        ln2_out_kernel<float><<<grid, 256, 0, s>>>(Z, stats, g2, be2, (float*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    return cudaGetLastError();
}

cudaError_t launch_pool(Act act, const float* Z, const float2* stats, const float* g2, const float* be2,
                        float* pooled, void* XL, int B, int T, int D, int Bcap, int nchunk, int cw, float eps,
                        int num_sms, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (T > kPoolMaxT) return cudaErrorNotSupported;
    const int grid = B < num_sms * 8 ? B : num_sms * 8;
    if (act == Act::BF16)
        pool_kernel<__nv_bfloat16><<<grid, kPoolThreads, 0, s>>>(Z, stats, g2, be2, pooled, (__nv_bfloat16*)XL, B, T,
                                                                  D, Bcap, nchunk, cw, eps);
    else
        pool_kernel<float><<<grid, kPoolThreads, 0, s>>>(Z, stats, g2, be2, pooled, (float*)XL, B, T, D, Bcap, nchunk,
                                                         cw, eps);
    return cudaGetLastError();
}

cudaError_t launch_rowstats(const float* Z, float2* stats, int B, int T, int D, int Bcap, int num_sms,
                            cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T * 32, 256, num_sms * 8);
    rowstats_kernel<<<grid, 256, 0, s>>>(Z, stats, B, T, D, Bcap);
    return cudaGetLastError();
}

cudaError_t launch_token_to_sample(Act act, const void* src, void* dst, int B, int T, int D, int Bcap,
                                   cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T * D, 256);
    if (act == Act::BF16)
        token_to_sample_kernel<__half, __nv_bfloat16><<<grid, 256, 0, s>>>((const __half*)src, (__nv_bfloat16*)dst,
                                                                           B, T, D, Bcap);
    else
        token_to_sample_kernel<float, float><<<grid, 256, 0, s>>>((const float*)src, (float*)dst, B, T, D, Bcap);
    return cudaGetLastError();
}

cudaError_t launch_token_mix(const void* X, void* Y, int B, int T, int D, int H, int esz, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T * D, 256);
    if (esz == 2)
        token_mix_kernel<uint16_t><<<grid, 256, 0, s>>>((const uint16_t*)X, (uint16_t*)Y, B, T, D, H);
    else if (esz == 4)
        token_mix_kernel<uint32_t><<<grid, 256, 0, s>>>((const uint32_t*)X, (uint32_t*)Y, B, T, D, H);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_pack_transpose(Act act, const void* in, void* out, int G, int R, int C, cudaStream_t s) {
    if (G <= 0 || R <= 0 || C <= 0) return cudaSuccess;
    dim3 grid((C + 31) / 32, (R + 31) / 32, G), block(32, 8);
    if (act == Act::BF16)
        transpose_kernel<__nv_bfloat16, __half><<<grid, block, 0, s>>>((const __nv_bfloat16*)in, (__half*)out, R, C);
    else
        transpose_kernel<float, float><<<grid, block, 0, s>>>((const float*)in, (float*)out, R, C);
    return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* in, float* out, int G, int R, int C, cudaStream_t s) {
    if (G <= 0 || R <= 0 || C <= 0) return cudaSuccess;
    dim3 grid((C + 31) / 32, (R + 31) / 32, G), block(32, 8);
    transpose_kernel<float, float><<<grid, block, 0, s>>>(in, out, R, C);
    return cudaGetLastError();
}

cudaError_t launch_to_f32(Act act, const void* in, float* out, size_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int grid = grid_for((long long)n, 256);
    if (act == Act::BF16)
        to_f32_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)in, out, n);
    else
        to_f32_kernel<float><<<grid, 256, 0, s>>>((const float*)in, out, n);
    return cudaGetLastError();
}

cudaError_t launch_debug_wait(const int* flag, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    debug_wait_kernel<<<1, 32, 0, s>>>(flag, err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace rm
