// UniMixing kernels ("UniMixer: A Unified Architecture for Scaling Laws in
// Recommendation Systems", section 4.3): the Sinkhorn-Knopp constraint of the
// mixing weights (Eq. 15), the per-block local step h_j = x_j WB_j (Eq. 13)
// and, after the global step Yt = WG H on the tensor cores, the residual +
// LN1 that feeds the per-token FFN (or a plain gather back to [B][T][D]).
//
// All three are memory-bound or tiny: the local step reads each sample once
// and writes H once (bs^2 multiply-adds per block of bs values, packed fp32x2
// FMAs on a bs x bs weight tile in shared memory); the row kernel reads X and
// Yt once and writes S once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "rm_common.cuh"
#include "rm_unimix.h"

namespace rm {
namespace {

// ---------------------------------------------------------------------------
// Sinkhorn-Knopp in the log domain
// ---------------------------------------------------------------------------
__global__ void sk_sym_kernel(const float* __restrict__ W, float* __restrict__ C, int count, int n, float scale) {
    const long long nn = (long long)n * n;
    const long long total = (long long)count * nn;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long c = idx / nn;
        const long long rem = idx - c * nn;
        const int i = (int)(rem / n), j = (int)(rem - (long long)i * n);
        const float* w = W + c * nn;
        C[idx] = (w[(long long)i * n + j] + w[(long long)j * n + i]) * scale;
    }
}

// out[row] = -LSE_j(C[row][j] + other[matrix(row)][j]), one warp per row.  C is
// symmetric, so the column step (a sum over i of C[i][j] + f[i]) is the same
// row reduction of row j.
__global__ void sk_lse_kernel(const float* __restrict__ C, int count, int n, const float* __restrict__ other,
                              float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)count * n;
    for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((long long)gridDim.x * blockDim.x) >> 5) {
        const long long c = row / n;
        const float* crow = C + row * n;
        const float* o = other + c * n;
        float m = -INFINITY, s = 0.f;
        for (int j = lane; j < n; j += 32) {
            const float x = crow[j] + o[j];
            if (x > m) {
                s = s * expf(m - x) + 1.f;
                m = x;
            } else {
                s += expf(x - m);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            const float M = fmaxf(m, m2);
            const float a = m == -INFINITY ? 0.f : s * expf(m - M);
            const float b = m2 == -INFINITY ? 0.f : s2 * expf(m2 - M);
            s = a + b;
            m = M;
        }
        if (lane == 0) out[row] = -(m + logf(s));
    }
}

__global__ void sk_fin_kernel(const float* __restrict__ C, const float* __restrict__ f, const float* __restrict__ g,
                              float* __restrict__ P32, __half* __restrict__ P16, int count, int n) {
    const long long nn = (long long)n * n;
    const long long total = (long long)count * nn;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long c = idx / nn;
        const long long rem = idx - c * nn;
        const int i = (int)(rem / n), j = (int)(rem - (long long)i * n);
        const float p = expf(C[idx] + f[c * n + i] + g[c * n + j]);
        P32[idx] = p;
        if (P16) P16[idx] = __float2half_rn(p);
    }
}

int grid_of(long long work, int threads) {
    long long g = (work + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > 152 * 32) g = 152 * 32;
    return (int)g;
}

// ---------------------------------------------------------------------------
// Local step
// ---------------------------------------------------------------------------
template <typename T> struct XLoad;
template <> struct XLoad<__nv_bfloat16> { static __device__ float at(const __nv_bfloat16* p) { return __bfloat162float(*p); } };
template <> struct XLoad<__half> { static __device__ float at(const __half* p) { return __half2float(*p); } };
template <> struct XLoad<float> { static __device__ float at(const float* p) { return *p; } };

__device__ __forceinline__ void store4(__half* p, float a, float b, float c, float d) {
    uint2 v;
    v.x = pack_f16x2(a, b);
    v.y = pack_f16x2(c, d);
    *reinterpret_cast<uint2*>(p) = v;
}
__device__ __forceinline__ void store4(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// bs % 4 == 0, bs <= 64.  CTA (sample tile, block j): WB_j and the tile's x_j
// rows in shared memory; thread (sg, rg) computes samples sg + k SG (k < SPT)
// x columns 4 rg .. 4 rg + 3, so a warp's stores cover consecutive samples'
// contiguous bs-wide runs of H's row j.
template <typename Tx, typename Top, int SPT>
__global__ void __launch_bounds__(256)
unimix_local_kernel(const Tx* __restrict__ X, long long x_stride, const float* __restrict__ WB, Top* __restrict__ H,
                    int B, int bs, long long Npitch, long long Npad) {
    extern __shared__ float smem[];
    const int j = blockIdx.y;
    const int rq = bs >> 2;
    const int SG = blockDim.x / rq;
    const int SB = SG * SPT;
    const int ldx = bs + 1;
    float* sW = smem;                   // [bs][bs]
    float* sX = smem + bs * bs;         // [SB][bs + 1]
    const float* wsrc = WB + (size_t)j * bs * bs;
    for (int e = threadIdx.x; e < bs * bs; e += blockDim.x) sW[e] = wsrc[e];
    const long long b0 = (long long)blockIdx.x * SB;
    for (int e = threadIdx.x; e < SB * bs; e += blockDim.x) {
        const int bb = e / bs, ss = e - bb * bs;
        const long long b = b0 + bb;
        sX[bb * ldx + ss] = b < B ? XLoad<Tx>::at(X + b * x_stride + (long long)j * bs + ss) : 0.f;
    }
    __syncthreads();
    const int rg = threadIdx.x % rq, sg = threadIdx.x / rq;
    if (sg < SG) {
        uint64_t a01[SPT], a23[SPT];
#pragma unroll
        for (int k = 0; k < SPT; ++k) a01[k] = a23[k] = 0ull;
        for (int s = 0; s < bs; ++s) {
            const float4 w = *reinterpret_cast<const float4*>(sW + s * bs + 4 * rg);
            const uint64_t w01 = f2_pack(w.x, w.y), w23 = f2_pack(w.z, w.w);
#pragma unroll
            for (int k = 0; k < SPT; ++k) {
                const uint64_t xv = f2_splat(sX[(sg + SG * k) * ldx + s]);
                a01[k] = f2_fma(xv, w01, a01[k]);
                a23[k] = f2_fma(xv, w23, a23[k]);
            }
        }
        Top* hrow = H + (size_t)j * Npitch;
#pragma unroll
        for (int k = 0; k < SPT; ++k) {
            const long long b = b0 + sg + SG * k;
            if (b < B) {
                float v0, v1, v2, v3;
                f2_unpack(a01[k], v0, v1);
                f2_unpack(a23[k], v2, v3);
                store4(hrow + b * bs + 4 * rg, v0, v1, v2, v3);
            }
        }
    }
    if (blockIdx.x == 0) {
        Top* hrow = H + (size_t)j * Npitch;
        for (long long n = (long long)B * bs + threadIdx.x; n < Npad; n += blockDim.x) hrow[n] = from_f32<Top>(0.f);
    }
}

// Any bs: one thread per output element.
template <typename Tx, typename Top>
__global__ void unimix_local_generic_kernel(const Tx* __restrict__ X, long long x_stride, const float* __restrict__ WB,
                                            Top* __restrict__ H, int B, int nb, int bs, long long Npitch,
                                            long long Npad) {
    const long long total = (long long)nb * Npad;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long j = idx / Npad;
        const long long n = idx - j * Npad;
        float acc = 0.f;
        if (n < (long long)B * bs) {
            const long long b = n / bs;
            const int r = (int)(n - b * bs);
            const Tx* x = X + b * x_stride + j * bs;
            const float* w = WB + j * bs * bs + r;
            for (int s = 0; s < bs; ++s) acc = fmaf(XLoad<Tx>::at(x + s), w[(size_t)s * bs], acc);
        }
        H[j * Npitch + n] = from_f32<Top>(acc);
    }
}

// ---------------------------------------------------------------------------
// Rows after the global step: one warp per (b, t) row of D values.  Element p
// = t D + d of sample b sits in Yt at (p / bs, b bs + p % bs); a lane walks its
// elements 32 apart, carrying (block, offset) forward instead of dividing.
// LN: S[t][b][:] = LN1(X + Y) in the operand type; otherwise Y in Tout.
// ---------------------------------------------------------------------------
template <typename Tx, typename Top, typename Tout, bool LN, int NI>
__global__ void __launch_bounds__(256)
unimix_rows_kernel(const Tx* __restrict__ X, const Top* __restrict__ Yt, Tout* __restrict__ out,
                   const float* __restrict__ g1, const float* __restrict__ be1, int B, int T, int D, int bs,
                   long long Npitch, int Bcap, float eps) {
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * T;
    for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((long long)gridDim.x * blockDim.x) >> 5) {
        const long long b = row / T;
        const int t = (int)(row - b * T);
        const long long p = (long long)t * D + lane;
        long long i = p / bs;
        int r = (int)(p - i * bs);
        const Top* ycol = Yt + b * bs;
        float v[NI];
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int d = lane + 32 * k;
            v[k] = 0.f;
            if (d < D) {
                float y = to_f32(ycol[i * Npitch + r]);
                if (LN) y += XLoad<Tx>::at(X + row * D + d);
                v[k] = y;
                sum += y;
            }
            r += 32;
            while (r >= bs) {
                r -= bs;
                ++i;
            }
        }
        if (LN) {
            const float mean = warp_sum(sum) / (float)D;
            float sq = 0.f;
#pragma unroll
            for (int k = 0; k < NI; ++k)
                if (lane + 32 * k < D) {
                    const float e = v[k] - mean;
                    sq += e * e;
                }
            const float rstd = rsqrtf(warp_sum(sq) / (float)D + eps);
            Tout* srow = out + ((size_t)t * Bcap + b) * D;
#pragma unroll
            for (int k = 0; k < NI; ++k) {
                const int d = lane + 32 * k;
                if (d < D) srow[d] = from_f32<Tout>(fmaf((v[k] - mean) * rstd, g1[d], be1[d]));
            }
        } else {
            Tout* yrow = out + row * D;
#pragma unroll
            for (int k = 0; k < NI; ++k) {
                const int d = lane + 32 * k;
                if (d < D) yrow[d] = from_f32<Tout>(v[k]);
            }
        }
    }
}

template <typename Tx, typename Top, typename Tout, bool LN>
cudaError_t launch_rows(const void* X, const void* Yt, void* out, const float* g1, const float* be1, int B, int T,
                        int D, int bs, long long Npitch, int Bcap, float eps, int num_sms, cudaStream_t s) {
    const long long rows = (long long)B * T;
    long long grid = (rows + 7) / 8;
    if (grid > (long long)num_sms * 16) grid = (long long)num_sms * 16;
    if (grid < 1) grid = 1;
#define RM_ROWS(NI)                                                                                            \
    unimix_rows_kernel<Tx, Top, Tout, LN, NI><<<(int)grid, 256, 0, s>>>(                                       \
        (const Tx*)X, (const Top*)Yt, (Tout*)out, g1, be1, B, T, D, bs, Npitch, Bcap, eps)
    const int ni = (D + 31) / 32;
    if (ni <= 8) RM_ROWS(8);
    else if (ni <= 16) RM_ROWS(16);
    else if (ni <= 32) RM_ROWS(32);
    else if (ni <= 48) RM_ROWS(48);
    else return cudaErrorNotSupported;
#undef RM_ROWS
    return cudaGetLastError();
}

template <typename Tx, typename Top>
cudaError_t launch_local_t(const void* X, long long x_stride, const float* WB, void* H, int B, int nb, int bs,
                           long long Npitch, long long Npad, cudaStream_t s) {
    if (bs % 4 == 0 && bs <= 64) {
        constexpr int SPT = 8;
        const int rq = bs / 4;
        const int SG = 256 / rq;
        const int threads = SG * rq;
        const int SB = SG * SPT;
        const size_t smem = ((size_t)bs * bs + (size_t)SB * (bs + 1)) * sizeof(float);
        auto k = unimix_local_kernel<Tx, Top, SPT>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const dim3 grid((unsigned)((B + SB - 1) / SB), (unsigned)nb);
        k<<<grid, threads, smem, s>>>((const Tx*)X, x_stride, WB, (Top*)H, B, bs, Npitch, Npad);
        return cudaGetLastError();
    }
    unimix_local_generic_kernel<Tx, Top><<<grid_of((long long)nb * Npad, 256), 256, 0, s>>>(
        (const Tx*)X, x_stride, WB, (Top*)H, B, nb, bs, Npitch, Npad);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sinkhorn(const float* W, int count, int n, float tau, int iters, float* C, float* f, float* g,
                            float* P32, void* P16, cudaStream_t s) {
    if (count <= 0 || n <= 0) return cudaSuccess;
    const long long total = (long long)count * n * n;
    sk_sym_kernel<<<grid_of(total, 256), 256, 0, s>>>(W, C, count, n, 0.5f / tau);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(f, 0, (size_t)count * n * sizeof(float), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(g, 0, (size_t)count * n * sizeof(float), s)) != cudaSuccess) return e;
    const int lse_grid = grid_of((long long)count * n * 32, 256);
    for (int it = 0; it < iters; ++it) {
        sk_lse_kernel<<<lse_grid, 256, 0, s>>>(C, count, n, g, f);   // rows
        sk_lse_kernel<<<lse_grid, 256, 0, s>>>(C, count, n, f, g);   // columns (C symmetric)
    }
    sk_fin_kernel<<<grid_of(total, 256), 256, 0, s>>>(C, f, g, P32, (__half*)P16, count, n);
    return cudaGetLastError();
}

cudaError_t launch_unimix_local(XType xt, Act act, const void* X, long long x_stride, const float* WB, void* H, int B,
                                int nb, int bs, long long Npitch, long long Npad, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act == Act::F32) {
        if (xt != XType::F32) return cudaErrorInvalidValue;
        return launch_local_t<float, float>(X, x_stride, WB, H, B, nb, bs, Npitch, Npad, s);
    }
    if (xt == XType::BF16) return launch_local_t<__nv_bfloat16, __half>(X, x_stride, WB, H, B, nb, bs, Npitch, Npad, s);
    if (xt == XType::F16) return launch_local_t<__half, __half>(X, x_stride, WB, H, B, nb, bs, Npitch, Npad, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_unimix_ln1(XType xt, Act act, const void* X, const void* Yt, void* S, const float* g1,
                              const float* be1, int B, int T, int D, int bs, long long Npitch, int Bcap, float eps,
                              int num_sms, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act == Act::F32) {
        if (xt != XType::F32) return cudaErrorInvalidValue;
        return launch_rows<float, float, float, true>(X, Yt, S, g1, be1, B, T, D, bs, Npitch, Bcap, eps, num_sms, s);
    }
    if (xt == XType::BF16)
        return launch_rows<__nv_bfloat16, __half, __half, true>(X, Yt, S, g1, be1, B, T, D, bs, Npitch, Bcap, eps,
                                                                num_sms, s);
    if (xt == XType::F16)
        return launch_rows<__half, __half, __half, true>(X, Yt, S, g1, be1, B, T, D, bs, Npitch, Bcap, eps, num_sms,
                                                         s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_unimix_gather(Act act, const void* Yt, void* Y, int B, int T, int D, int bs, long long Npitch,
                                 int num_sms, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act == Act::F32)
        return launch_rows<float, float, float, false>(nullptr, Yt, Y, nullptr, nullptr, B, T, D, bs, Npitch, B, 0.f,
                                                       num_sms, s);
    return launch_rows<__half, __half, __nv_bfloat16, false>(nullptr, Yt, Y, nullptr, nullptr, B, T, D, bs, Npitch, B,
                                                             0.f, num_sms, s);
}

}  // namespace rm
