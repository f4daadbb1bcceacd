// CUDA-core per-token FFN GEMMs.  Used for the float32 path (the tensor
// cores have no exact-fp32 MMA kind) and for shapes the tcgen05 kernels do
// not tile.  Grouped: grid.z = token t, each token with its own weights.
// Operands are float32 (float32 contexts) or fp16 (bf16 contexts), as on the
// tensor-core path; accumulation is float32.
//
// "RankMixer: Scaling Up Ranking Models in Industrial Recommenders", section
// 3.3.2 Eq. 6-7: u_t = s_t W1_t + b1_t, a_t = Gelu(u_t), v_t = a_t W2_t + b2_t.
#include "rm_common.cuh"
#include "rm_internal.h"

namespace rm {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

enum { EPI_GELU = 1, EPI_RESID = 2 };

// out[t][m][n] = epi(sum_k A[t][m][k] * W[t][n][k] + bias[t][n]).
// A token-major [T][Bcap][K], W [T][N][K], outputs token-major [T][Bcap][N] in
// the operand type (EPI_GELU: hidden activations, EPI_RESID: Z = . + S).
template <typename Tin, int EPI>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const Tin* __restrict__ A, const Tin* __restrict__ W, const float* __restrict__ bias,
                 void* __restrict__ out, const Tin* __restrict__ resid, int M, int N, int K, int Bcap) {
    __shared__ float As[TK][TM + 4];
    __shared__ float Ws[TK][TN + 4];
    const int t = blockIdx.z;
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const Tin* At = A + (size_t)t * Bcap * K;
    const Tin* Wt = W + (size_t)t * N * K;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    const int lr = threadIdx.x >> 2;        // 0..63: tile row loaded by this thread
    const int lk = (threadIdx.x & 3) * 4;   // 0,4,8,12: first k of its 4 elements
    for (int k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = k0 + lk + e;
            const int m = m0 + lr, n = n0 + lr;
            As[lk + e][lr] = (m < M && k < K) ? to_f32(At[(size_t)m * K + k]) : 0.f;
            Ws[lk + e][lr] = (n < N && k < K) ? to_f32(Wt[(size_t)n * K + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float a[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n >= N) continue;
            const size_t o = ((size_t)t * Bcap + m) * N + n;
            const float u = acc[i][j] + bias[(size_t)t * N + n];
            if (EPI == EPI_GELU) {
                reinterpret_cast<Tin*>(out)[o] = from_f32<Tin>(gelu_erf(u));
            } else {
                reinterpret_cast<Tin*>(out)[o] = from_f32<Tin>(u + to_f32(resid[o]));
            }
        }
    }
}

template <typename Tin, int EPI>
cudaError_t launch(const void* A, const void* W, const float* bias, void* out, const void* resid, int M, int N, int K,
                   int T, int Bcap, cudaStream_t s) {
    dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM, T);
    gemm_simt_kernel<Tin, EPI><<<grid, 256, 0, s>>>((const Tin*)A, (const Tin*)W, bias, out, (const Tin*)resid, M, N,
                                                    K, Bcap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1_simt(Act act, const void* S, const void* W1p, const float* b1, void* Hid, int B, int T,
                              int D, int F, int Bcap, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act == Act::BF16) return launch<__half, EPI_GELU>(S, W1p, b1, Hid, nullptr, B, F, D, T, Bcap, s);
    return launch<float, EPI_GELU>(S, W1p, b1, Hid, nullptr, B, F, D, T, Bcap, s);
}

cudaError_t launch_gemm2_simt(Act act, const void* Hid, const void* W2p, const float* b2, const void* S, void* Z,
                              int B, int T, int D, int F, int Bcap, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act == Act::BF16) return launch<__half, EPI_RESID>(Hid, W2p, b2, Z, S, B, D, F, T, Bcap, s);
    return launch<float, EPI_RESID>(Hid, W2p, b2, Z, S, B, D, F, T, Bcap, s);
}

}  // namespace rm
