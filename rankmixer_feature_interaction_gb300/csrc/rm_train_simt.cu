// SIMT path of the backward-pass GEMMs (any shape, float32 or fp16 operands):
// 64 x 64 output tiles, 16-deep k slices staged in shared memory as float32,
// 4 x 4 outputs per thread.  The same products and epilogues as the
// tensor-core path (see rm_train.h); used for float32 contexts, for shapes the
// tensor-core kernel does not take, and as its cross-check in the tests.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rm_common.cuh"
#include "rm_train.h"
#include "rm_train_math.cuh"

namespace rm {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

// Element (r, k) of an operand of group g (r: the M or N index), 0 outside.
template <typename Top>
__device__ __forceinline__ float op_at(const TOperand& o, int g, int r, int k, int r_lim, int k_lim) {
    if (r >= r_lim || k >= k_lim) return 0.f;
    const Top* p = reinterpret_cast<const Top*>(o.ptr) + (size_t)g * (size_t)o.gpitch;
    const size_t ld = o.ld ? (size_t)o.ld : (size_t)o.inner;
    if (o.mn) {
        if (k >= o.outer || r >= o.inner) return 0.f;
        return to_f32(p[(size_t)k * ld + r]);
    }
    if (r >= o.outer || k >= o.inner) return 0.f;
    return to_f32(p[(size_t)r * ld + k]);
}

template <typename Top, typename Taux, int EPI>
__global__ void __launch_bounds__(256)
train_gemm_simt_kernel(const TrainGemm g) {
    __shared__ float sA[TK][TM + 1];
    __shared__ float sB[TK][TN + 1];
    const int grp = blockIdx.z;
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += TK) {
        for (int i = threadIdx.x; i < TM * TK; i += 256) {
            const int kk = i % TK, rr = i / TK;
            sA[kk][rr] = op_at<Top>(g.a, grp, m0 + rr, k0 + kk, g.M, g.K);
            sB[kk][rr] = op_at<Top>(g.b, grp, n0 + rr, k0 + kk, g.N, g.K);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = sA[kk][ty + 16 * i];
                bv[i] = sB[kk][tx + 16 * i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    const float inv_s = g.inv_scale ? g.inv_scale[grp] : 1.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= g.m_valid) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n >= g.N) continue;
            const size_t off = (size_t)grp * (size_t)g.c_gpitch + (size_t)m * (g.c_ld ? (size_t)g.c_ld : (size_t)g.N) + n;
            const float raw = acc[i][j];
            const float v = raw * inv_s;
            if (EPI == TE_GELU2) {
                const GeluPair x = gelu_with_grad(v + g.bias[(size_t)grp * g.N + n]);
                reinterpret_cast<Top*>(g.c0)[off] = from_f32<Top>(x.value);
                reinterpret_cast<Taux*>(g.c1)[off] = from_f32<Taux>(x.grad);
            } else if (EPI == TE_RESID) {
                const float r = to_f32(reinterpret_cast<const Top*>(g.r)[off]);
                reinterpret_cast<Taux*>(g.c0)[off] = from_f32<Taux>(v + g.bias[(size_t)grp * g.N + n] + r);
            } else if (EPI == TE_DGELU) {      // stays in the scaled domain
                const float gp = to_f32(reinterpret_cast<const Taux*>(g.r)[off]);
                reinterpret_cast<Top*>(g.c0)[off] = from_f32<Top>(raw * gp);
            } else if (EPI == TE_DRESID) {
                reinterpret_cast<float*>(g.c0)[off] = v + reinterpret_cast<const float*>(g.r)[off];
            } else if (EPI == TE_BIAS_IO) {      // the caller dtype: float, or bf16 for fp16-operand contexts
                const float o = v + g.bias[(size_t)grp * g.N + n];
                if constexpr (std::is_same_v<Top, float>)
                    reinterpret_cast<float*>(g.c0)[off] = o;
                else
                    reinterpret_cast<__nv_bfloat16*>(g.c0)[off] = __float2bfloat16_rn(o);
            } else if (EPI == TE_F16) {        // the operand type (fp16, or float for float32 contexts)
                reinterpret_cast<Top*>(g.c0)[off] = from_f32<Top>(v);
            } else if (EPI == TE_F16T) {       // column n = b bs + r of row m -> Y[b][m bs + r]
                const int b = n / g.um_bs;
                if (b < g.um_B)
                    reinterpret_cast<Top*>(g.c0)[(size_t)b * g.um_L + (size_t)m * g.um_bs + (n - b * g.um_bs)] =
                        from_f32<Top>(v);
            } else {
                reinterpret_cast<float*>(g.c0)[off] = v;
            }
        }
    }
}

// out[g][n] = inv_scale[g] * sum over m < rows of C[g][m][n] (C of type T, group pitch gpitch).
template <typename T>
__global__ void colsum_kernel(const T* __restrict__ C, long long gpitch, int rows, int N,
                              const float* __restrict__ inv_scale, float* __restrict__ out) {
    const int grp = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const T* p = C + (size_t)grp * (size_t)gpitch + n;   // rows N apart (TE_DGELU outputs are dense)
    const float inv_s = inv_scale ? inv_scale[grp] : 1.0f;
    float s = 0.f;
    for (int m = 0; m < rows; ++m) s = fmaf(to_f32(p[(size_t)m * N]), inv_s, s);
    out[(size_t)grp * N + n] = s;
}

template <typename Top, typename Taux>
cudaError_t run_simt(int epi, const TrainGemm& g, cudaStream_t s) {
    const dim3 grid((g.N + TN - 1) / TN, (g.m_valid + TM - 1) / TM, g.G);
    switch (epi) {
        case TE_GELU2: train_gemm_simt_kernel<Top, Taux, TE_GELU2><<<grid, 256, 0, s>>>(g); break;
        case TE_RESID: train_gemm_simt_kernel<Top, Taux, TE_RESID><<<grid, 256, 0, s>>>(g); break;
        case TE_DGELU: train_gemm_simt_kernel<Top, Taux, TE_DGELU><<<grid, 256, 0, s>>>(g); break;
        case TE_DRESID: train_gemm_simt_kernel<Top, Taux, TE_DRESID><<<grid, 256, 0, s>>>(g); break;
        case TE_F32: train_gemm_simt_kernel<Top, Taux, TE_F32><<<grid, 256, 0, s>>>(g); break;
        case TE_BIAS_IO: train_gemm_simt_kernel<Top, Taux, TE_BIAS_IO><<<grid, 256, 0, s>>>(g); break;
        case TE_F16: train_gemm_simt_kernel<Top, Taux, TE_F16><<<grid, 256, 0, s>>>(g); break;
        case TE_F16T: train_gemm_simt_kernel<Top, Taux, TE_F16T><<<grid, 256, 0, s>>>(g); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || epi != TE_DGELU || g.colpart == nullptr) return e;
    const dim3 cgrid((g.N + 255) / 256, g.G);
    colsum_kernel<Top><<<cgrid, 256, 0, s>>>(reinterpret_cast<const Top*>(g.c0), g.c_gpitch, g.m_valid, g.N,
                                              g.inv_scale, g.colpart);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_train_gemm_simt(Act act, int epi, const TrainGemm& g, cudaStream_t s) {
    if (g.G <= 0 || g.m_valid <= 0 || g.N <= 0) return cudaSuccess;
    if (act == Act::F32) return run_simt<float, float>(epi, g, s);
    return run_simt<__half, __half>(epi, g, s);
}

}  // namespace rm
