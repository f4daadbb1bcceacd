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

}  // namespace rm
