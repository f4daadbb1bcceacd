// Prediction head on the pooled output ("RankMixer 详解（1）" sections 5.1-5.2):
//   z = o w + b,  p = sigmoid(z),  l = -y log p - (1 - y) log(1 - p),
//   dl/dz = p - y,  dl/do = (p - y) w.
// One warp per sample: the dot product over D with 16-byte loads when D allows,
// then lane 0 forms p and the loss; the gradient row is written by the whole
// warp.  log p = -softplus(-z) and log(1 - p) = -softplus(z) keep the loss
// finite for any z.
#include <cuda_runtime.h>

#include "rm_common.cuh"
#include "rm_train.h"

namespace rm {
namespace {

__device__ __forceinline__ float softplus_f(float x) {
    return x > 0.f ? x + log1pf(__expf(-x)) : log1pf(__expf(x));
}

__global__ void __launch_bounds__(256)
head_kernel(const float* __restrict__ O, const float* __restrict__ w, float b, const float* __restrict__ y,
            float* __restrict__ p_out, float* __restrict__ loss_out, float* __restrict__ dO, float gscale, int B,
            int D) {
    const int lane = threadIdx.x & 31;
    const bool vec = (D & 3) == 0;
    for (int i = blockIdx.x * 8 + (threadIdx.x >> 5); i < B; i += gridDim.x * 8) {
        const float* o = O + (size_t)i * D;
        float acc = 0.f;
        if (vec) {
            for (int j = 4 * lane; j < D; j += 128) {
                const float4 a = *reinterpret_cast<const float4*>(o + j);
                const float4 c = __ldg(reinterpret_cast<const float4*>(w + j));
                acc = fmaf(a.x, c.x, fmaf(a.y, c.y, fmaf(a.z, c.z, fmaf(a.w, c.w, acc))));
            }
        } else {
            for (int j = lane; j < D; j += 32) acc = fmaf(o[j], __ldg(w + j), acc);
        }
        const float z = warp_sum(acc) + b;
        const float p = 1.0f / (1.0f + __expf(-z));
        if (lane == 0 && p_out) p_out[i] = p;
        if (!y) continue;
        const float yi = y[i];
        if (lane == 0 && loss_out) loss_out[i] = yi * softplus_f(-z) + (1.0f - yi) * softplus_f(z);
        if (dO) {
            const float g = gscale * (p - yi);
            float* d = dO + (size_t)i * D;
            for (int j = lane; j < D; j += 32) d[j] = g * __ldg(w + j);
        }
    }
}

}  // namespace

cudaError_t launch_head(const float* pooled, const float* w, float b, const float* y, float* p, float* loss, float* dO,
                        float gscale, int B, int D, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    int grid = (B + 7) / 8;
    if (grid > 4096) grid = 4096;
    head_kernel<<<grid, 256, 0, s>>>(pooled, w, b, y, p, loss, dO, gscale, B, D);
    return cudaGetLastError();
}

// ---- tokenization backward helpers ------------------------------------------------
// Per-token scale of a sample-major gradient G [B][T][D] (as grad_scale does for
// the token-major dZ): part[t][x] = the largest |G[b][t][:]| over CTA x's
// samples, then s_t = 2^(9 - e) with 2^e >= max_x part[t][x], inv[t] = 1 / s_t
// and Gh = fp16(s_t G).
namespace {
__global__ void __launch_bounds__(256)
token_absmax_kernel(const float* __restrict__ G, float* __restrict__ part, int B, int T, int D) {
    __shared__ float red[256];
    const int t = blockIdx.y;
    float m = 0.f;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        const float* g = G + ((size_t)b * T + t) * D;
        for (int k = threadIdx.x; k < D; k += 256) m = fmaxf(m, fabsf(g[k]));
    }
    red[threadIdx.x] = m;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + o]);
        __syncthreads();
    }
    if (threadIdx.x == 0) part[(size_t)t * gridDim.x + blockIdx.x] = red[0];
}

__global__ void __launch_bounds__(256)
token_scale_convert_kernel(const float* __restrict__ G, const float* __restrict__ part, int nparts,
                           float* __restrict__ inv_scale, __half* __restrict__ Gh, int B, int T, int D) {
    __shared__ float sc;
    const int t = blockIdx.y;
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int i = 0; i < nparts; ++i) m = fmaxf(m, part[(size_t)t * nparts + i]);
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
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        const size_t o = ((size_t)b * T + t) * D;
        for (int k = threadIdx.x; k < D; k += 256) Gh[o + k] = __float2half_rn(sat_f16(G[o + k] * s));
    }
}

// db[t][k] = sum over b of G[b][t][k] (sample-major G), fixed order.
__global__ void token_colsum_kernel(const float* __restrict__ G, float* __restrict__ db, int B, int T, int D) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * D) return;
    const int t = (int)(i / D), k = (int)(i - (long long)t * D);
    float s = 0.f;
    for (int b = 0; b < B; ++b) s += G[((size_t)b * T + t) * D + k];
    db[i] = s;
}
}  // namespace

cudaError_t launch_token_grad_scale(const float* G, float* part, int nparts, float* inv_scale, void* Gh, int B, int T,
                                    int D, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const dim3 grid(nparts, T);
    token_absmax_kernel<<<grid, 256, 0, s>>>(G, part, B, T, D);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    token_scale_convert_kernel<<<grid, 256, 0, s>>>(G, part, nparts, inv_scale, (__half*)Gh, B, T, D);
    return cudaGetLastError();
}

cudaError_t launch_token_colsum(const float* G, float* db, int B, int T, int D, cudaStream_t s) {
    const long long n = (long long)T * D;
    if (n <= 0) return cudaSuccess;
    token_colsum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(G, db, B, T, D);
    return cudaGetLastError();
}

}  // namespace rm
