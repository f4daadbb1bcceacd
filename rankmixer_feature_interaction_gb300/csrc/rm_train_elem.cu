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
constexpr int kLn2Rows = 32;                 // rows (samples) of one token per CTA
constexpr int kLn2MaxCols = 3072 / kLn2Threads;
constexpr int kLn1Threads = 512;
constexpr int kLn1MaxCols = 3072 / kLn1Threads;
constexpr int kLn1SmemLimit = 200 * 1024;    // bytes of dY a CTA may hold in shared memory

// Element k of the residual row y = Mix(X)[t] + X[t] of one sample:
// Mix(X)[t][c q + r] = X[c][t q + r].
template <typename Tx>
__device__ __forceinline__ float mixed_row_elem(const Tx* __restrict__ Xb, int t, int k, int q, int D) {
    const int c = k / q, r = k - (k / q) * q;
    return to_f32(Xb[(size_t)c * D + (size_t)t * q + r]) + to_f32(Xb[(size_t)t * D + k]);
}

// Mean and 1 / sqrt(var + eps) of y = Mix(X)[t] + X[t] (called by a full warp).
template <typename Tx>
__device__ __forceinline__ void mixed_row_stats(const Tx* __restrict__ Xb, int t, int q, int D, float eps, int lane,
                                                float& mean, float& rstd) {
    const float shift = mixed_row_elem(Xb, t, 0, q, D);     // shifted sums keep the variance accurate
    float s1 = 0.f, s2 = 0.f;
    for (int k = lane; k < D; k += 32) {
        const float d = mixed_row_elem(Xb, t, k, q, D) - shift;
        s1 += d;
        s2 = fmaf(d, d, s2);
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    const float dm = s1 / (float)D;
    mean = shift + dm;
    rstd = rsqrtf(fmaxf(s2 / (float)D - dm * dm, 0.f) + eps);
}

// ---- LN1 recompute ---------------------------------------------------------------
template <typename Tx, typename Top>
__global__ void __launch_bounds__(256)
ln1_recompute_kernel(const Tx* __restrict__ X, Top* __restrict__ S, const float* __restrict__ g1,
                     const float* __restrict__ be1, int B, int T, int D, int Bcap, float eps) {
    const int lane = threadIdx.x & 31;
    const int q = D / T;
    const long long rows = (long long)B * T;
    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += (long long)gridDim.x * 8) {
        const int b = (int)(row / T), t = (int)(row - (long long)b * T);
        const Tx* Xb = X + (size_t)b * T * D;
        float mean, rstd;
        mixed_row_stats(Xb, t, q, D, eps, lane, mean, rstd);
        Top* out = S + ((size_t)t * Bcap + b) * D;
        for (int k = lane; k < D; k += 32)
            out[k] = from_f32<Top>(fmaf(g1[k], (mixed_row_elem(Xb, t, k, q, D) - mean) * rstd, be1[k]));
    }
}

// ---- LN2 backward ----------------------------------------------------------------
template <typename Tz>
__global__ void __launch_bounds__(kLn2Threads)
ln2_backward_kernel(const Tz* __restrict__ Z, const float* __restrict__ G, const float* __restrict__ g2,
                    float* __restrict__ dZ, float* __restrict__ part_db2, float* __restrict__ part_dg2,
                    float* __restrict__ part_dbe2, float* __restrict__ part_max, int B, int T, int D, int Bcap,
                    float eps) {
    __shared__ float4 st[kLn2Rows];          // (mean, rstd, mean(q), mean(q zhat)) per row
    __shared__ float wmax[kLn2Threads / 32];
    const int t = blockIdx.y, blk = blockIdx.x, nblk = gridDim.x;
    const int b0 = blk * kLn2Rows;
    const int nrows = min(kLn2Rows, B - b0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < nrows; i += kLn2Threads / 32) {
        const int b = b0 + i;
        const Tz* z = Z + ((size_t)t * Bcap + b) * D;
        const float* gr = G + ((size_t)b * T + t) * D;
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
        if (lane == 0) st[i] = make_float4(mean, rstd, mq / (float)D, mqz / (float)D);
    }
    __syncthreads();
    float adb[kLn2MaxCols], adg[kLn2MaxCols], adbe[kLn2MaxCols];
#pragma unroll
    for (int c = 0; c < kLn2MaxCols; ++c) adb[c] = adg[c] = adbe[c] = 0.f;
    float amax = 0.f;
    for (int i = 0; i < nrows; ++i) {
        const float4 s = st[i];
        const int b = b0 + i;
        const Tz* z = Z + ((size_t)t * Bcap + b) * D;
        const float* gr = G + ((size_t)b * T + t) * D;
        float* dz = dZ + ((size_t)t * Bcap + b) * D;
#pragma unroll
        for (int c = 0; c < kLn2MaxCols; ++c) {
            const int k = threadIdx.x + c * kLn2Threads;
            if (k < D) {
                const float zh = (to_f32(z[k]) - s.x) * s.y;
                const float gk = gr[k];
                const float d = (gk * g2[k] - s.z - zh * s.w) * s.y;
                dz[k] = d;
                amax = fmaxf(amax, fabsf(d));
                adb[c] += d;
                adg[c] = fmaf(gk, zh, adg[c]);
                adbe[c] += gk;
            }
        }
    }
    const size_t prow = ((size_t)t * nblk + blk) * D;
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
        part_max[(size_t)t * nblk + blk] = m;
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
template <typename Tx, bool SMEM_DY>
__global__ void __launch_bounds__(kLn1Threads)
ln1_mix_backward_kernel(const Tx* __restrict__ X, const float* __restrict__ dS, const float* __restrict__ g1,
                        float* __restrict__ dX, float* __restrict__ part_dg1, float* __restrict__ part_dbe1,
                        float* __restrict__ scratch, int B, int T, int D, int Bcap, float eps) {
    extern __shared__ float4 smem4[];
    float4* st = smem4;                                      // [T] (mean, rstd, mean(q), mean(q yhat))
    float* dY = SMEM_DY ? reinterpret_cast<float*>(smem4 + T) : scratch + (size_t)blockIdx.x * T * D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = D / T;
    float adg[kLn1MaxCols], adbe[kLn1MaxCols];
#pragma unroll
    for (int c = 0; c < kLn1MaxCols; ++c) adg[c] = adbe[c] = 0.f;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        const Tx* Xb = X + (size_t)b * T * D;
        for (int t = warp; t < T; t += kLn1Threads / 32) {
            float mean, rstd;
            mixed_row_stats(Xb, t, q, D, eps, lane, mean, rstd);
            const float* ds = dS + ((size_t)t * Bcap + b) * D;
            float mq = 0.f, mqy = 0.f;
            for (int k = lane; k < D; k += 32) {
                const float qk = ds[k] * g1[k];
                mq += qk;
                mqy = fmaf(qk, (mixed_row_elem(Xb, t, k, q, D) - mean) * rstd, mqy);
            }
            mq = warp_sum(mq);
            mqy = warp_sum(mqy);
            if (lane == 0) st[t] = make_float4(mean, rstd, mq / (float)D, mqy / (float)D);
        }
        __syncthreads();
        for (int t = 0; t < T; ++t) {
            const float4 s = st[t];
            const float* ds = dS + ((size_t)t * Bcap + b) * D;
#pragma unroll
            for (int c = 0; c < kLn1MaxCols; ++c) {
                const int k = threadIdx.x + c * kLn1Threads;
                if (k < D) {
                    const float yh = (mixed_row_elem(Xb, t, k, q, D) - s.x) * s.y;
                    const float dk = ds[k];
                    dY[(size_t)t * D + k] = (dk * g1[k] - s.z - yh * s.w) * s.y;
                    adg[c] = fmaf(dk, yh, adg[c]);
                    adbe[c] += dk;
                }
            }
        }
        __syncthreads();
        // dX[t][c q + r] = dY[t][c q + r] + dY[c][t q + r]
        float* out = dX + (size_t)b * T * D;
        const int n = T * D;
        for (int i = threadIdx.x; i < n; i += kLn1Threads) {
            const int t = i / D, k = i - (i / D) * D;
            const int c = k / q, r = k - (k / q) * q;
            out[i] = dY[i] + dY[(size_t)c * D + (size_t)t * q + r];
        }
        __syncthreads();
    }
#pragma unroll
    for (int c = 0; c < kLn1MaxCols; ++c) {
        const int k = threadIdx.x + c * kLn1Threads;
        if (k < D) {
            part_dg1[(size_t)blockIdx.x * D + k] = adg[c];
            part_dbe1[(size_t)blockIdx.x * D + k] = adbe[c];
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

__global__ void pool_backward_kernel(const float* __restrict__ dP, float* __restrict__ G, int B, int T, int D) {
    const long long n = (long long)B * T * D;
    const float inv = 1.0f / (float)T;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long b = i / ((long long)T * D);
        const int k = (int)(i % D);
        G[i] = dP[b * D + k] * inv;
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

size_t ln1_smem_bytes(int T, int D) { return (size_t)T * sizeof(float4) + (size_t)T * D * sizeof(float); }

}  // namespace

cudaError_t launch_ln1_recompute(Act act, bool x_f32, const void* X, void* S, const float* g1, const float* be1,
                                 int B, int T, int D, int Bcap, float eps, int num_sms, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T, 8, num_sms * 8);
    if (act == Act::F32)
        ln1_recompute_kernel<float, float><<<grid, 256, 0, s>>>((const float*)X, (float*)S, g1, be1, B, T, D, Bcap,
                                                                 eps);
    else if (x_f32)
        ln1_recompute_kernel<float, __half><<<grid, 256, 0, s>>>((const float*)X, (__half*)S, g1, be1, B, T, D,
                                                                  Bcap, eps);
    else
        ln1_recompute_kernel<__nv_bfloat16, __half><<<grid, 256, 0, s>>>((const __nv_bfloat16*)X, (__half*)S, g1,
                                                                          be1, B, T, D, Bcap, eps);
    return cudaGetLastError();
}

int ln2_bwd_row_block() { return kLn2Rows; }

cudaError_t launch_ln2_backward(Act act, const void* Z, const float* G, const float* g2, float* dZ, float* part_db2,
                                float* part_dg2, float* part_dbe2, float* part_max, int B, int T, int D, int Bcap,
                                float eps, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (D > kLn2MaxCols * kLn2Threads) return cudaErrorNotSupported;
    const dim3 grid((B + kLn2Rows - 1) / kLn2Rows, T);
    if (act == Act::F32)
        ln2_backward_kernel<float><<<grid, kLn2Threads, 0, s>>>((const float*)Z, G, g2, dZ, part_db2, part_dg2,
                                                                 part_dbe2, part_max, B, T, D, Bcap, eps);
    else
        ln2_backward_kernel<__half><<<grid, kLn2Threads, 0, s>>>((const __half*)Z, G, g2, dZ, part_db2, part_dg2,
                                                                  part_dbe2, part_max, B, T, D, Bcap, eps);
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

int ln1_bwd_grid(int B, int num_sms) { return B < num_sms ? (B < 1 ? 1 : B) : num_sms; }

bool ln1_bwd_needs_scratch(int T, int D) { return ln1_smem_bytes(T, D) > (size_t)kLn1SmemLimit; }

cudaError_t launch_ln1_mix_backward(Act act, bool x_f32, const void* X, const float* dS, const float* g1, float* dX,
                                    float* part_dg1, float* part_dbe1, float* scratch, int B, int T, int D, int Bcap,
                                    float eps, int grid, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (D > kLn1MaxCols * kLn1Threads) return cudaErrorNotSupported;
    const bool smem = !ln1_bwd_needs_scratch(T, D);
    if (!smem && scratch == nullptr) return cudaErrorInvalidValue;
    const size_t bytes = smem ? ln1_smem_bytes(T, D) : (size_t)T * sizeof(float4);
#define RM_LN1B(TX, SM)                                                                                        \
    do {                                                                                                       \
        auto k = ln1_mix_backward_kernel<TX, SM>;                                                              \
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);      \
        if (e != cudaSuccess) return e;                                                                        \
        k<<<grid, kLn1Threads, bytes, s>>>((const TX*)X, dS, g1, dX, part_dg1, part_dbe1, scratch, B, T, D,    \
                                           Bcap, eps);                                                         \
    } while (0)
    if (act == Act::F32 || x_f32) {
        if (smem) RM_LN1B(float, true); else RM_LN1B(float, false);
    } else {
        if (smem) RM_LN1B(__nv_bfloat16, true); else RM_LN1B(__nv_bfloat16, false);
    }
#undef RM_LN1B
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
    pool_backward_kernel<<<grid_for((long long)B * T * D, 256, 4096), 256, 0, s>>>(dpooled, G, B, T, D);
    return cudaGetLastError();
}

cudaError_t launch_debug_gelu_grad(const float* u, float* out, long long n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    debug_gelu_grad_kernel<<<grid_for(n, 256, 4096), 256, 0, s>>>(u, out, n);
    return cudaGetLastError();
}

}  // namespace rm
