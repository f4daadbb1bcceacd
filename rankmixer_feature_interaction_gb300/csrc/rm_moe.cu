// Sparse-MoE per-token FFN with ReLU routing.
//
// "RankMixer: Scaling Up Ranking Models in Industrial Recommenders", section
// 3.4 Eq. 10: for token t the inference router h_t gives gates
// G_{t,e} = ReLU(h_t(s_t)) and v_t = sum_e G_{t,e} e_{t,e}(s_t), every expert
// e_{t,e} a two-layer GELU FFN owned by token t alone.  The number of active
// experts varies per token and sample; experts with G = 0 contribute exactly
// zero and are skipped.
//
// Pipeline (all on the launch stream, no host synchronisation):
//   1 router      one warp per (b, t): G = ReLU(s Wg_t + bg_t)
//   2 count       one CTA per (t, e): number of samples with G > 0
//   3 prefix      one thread: row offsets, 128-row tile prefixes per launch
//   4 fill        one CTA per (t, e): ascending list of the active samples
//   5 gather      packed rows Sg[off(t,e) + i] = S[b_i, t]   (fp16 operands for bf16 contexts)
//   6 expert L1   variable-size grouped GEMM + bias + GELU -> Hm (packed rows)
//   7 expert L2   one launch per expert index e (fixed order e = 0..E-1):
//                 V[b, t] += G * (Hm W2_{t,e} + b2_{t,e})
// The fixed order of step 7 makes the float32 sum over experts deterministic.
#include <vector>

#include "rm_common.cuh"
#include "rm_internal.h"
#include "rm_moe.h"

namespace rm {

// tcgen05 launchers (rm_gemm_tc.cu)
cudaError_t launch_moe_gemm1_tc(const void* Sg, long long rows_total, const void* W1p, const float* b1, void* Hm,
                                int groups, int D, int Fe, const int* g_count, const int* g_off,
                                const int* tile_prefix, int num_sms, int* err, unsigned long long timeout_ns,
                                cudaStream_t s);
cudaError_t launch_moe_gemm2_tc(const void* Hm, long long rows_total, const void* W2p, const float* b2, int T, int E,
                                int e, int D, int Fe, const int* g_count, const int* g_off, const int* tile_prefix_e,
                                const int* row_sample, const float* gates, float* V, long long v_sb, long long v_st,
                                int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s);

namespace {

constexpr unsigned long long kMoeWaitTimeoutNs = 2000000000ull;

// ---- 1: router -------------------------------------------------------------------
template <typename Tact>
__global__ void router_kernel(const Tact* __restrict__ S, long long s_sb, long long s_st, const float* __restrict__ Wg,
                              const float* __restrict__ bg, float* __restrict__ gates, int B, int T, int D, int E) {
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = wid; r < (long long)B * T; r += nw) {
        const int b = (int)(r / T), t = (int)(r % T);
        const Tact* s = S + b * s_sb + t * s_st;
        for (int e = 0; e < E; ++e) {
            const float* w = Wg + ((size_t)t * E + e) * D;
            float acc = 0.f;
            for (int j = lane; j < D; j += 32) acc = fmaf(to_f32(s[j]), w[j], acc);
            acc = warp_sum(acc);
            if (lane == 0) gates[((size_t)b * T + t) * E + e] = fmaxf(acc + bg[(size_t)t * E + e], 0.f);
        }
    }
}

// ---- 2: per-(t, e) active count -------------------------------------------------
__global__ void count_kernel(const float* __restrict__ gates, int* __restrict__ counts, int B, int T, int E) {
    __shared__ int s_cnt;
    const int g = blockIdx.x;
    const int t = g / E, e = g % E;
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    int c = 0;
    for (int b = threadIdx.x; b < B; b += blockDim.x) c += gates[((size_t)b * T + t) * E + e] > 0.f;
    atomicAdd(&s_cnt, c);
    __syncthreads();
    if (threadIdx.x == 0) counts[g] = s_cnt;
}

// ---- 3: offsets and tile prefixes ---------------------------------------------------
// offsets[g] over g = t E + e; tile_prefix[0 .. G] over the same order (expert layer 1);
// tile_prefix[G + 1 + e (T + 1) + t] over t for fixed e (expert layer 2, one launch per e).
__global__ void prefix_kernel(const int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ tile_prefix,
                              int T, int E) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const int G = T * E;
    int off = 0, tp = 0;
    for (int g = 0; g < G; ++g) {
        offsets[g] = off;
        tile_prefix[g] = tp;
        off += counts[g];
        tp += (counts[g] + 127) / 128;
    }
    offsets[G] = off;
    tile_prefix[G] = tp;
    for (int e = 0; e < E; ++e) {
        int* p = tile_prefix + G + 1 + e * (T + 1);
        int acc = 0;
        for (int t = 0; t < T; ++t) {
            p[t] = acc;
            acc += (counts[t * E + e] + 127) / 128;
        }
        p[T] = acc;
    }
}

// ---- 4: ordered compaction -------------------------------------------------------
__global__ void __launch_bounds__(256) fill_kernel(const float* __restrict__ gates, const int* __restrict__ offsets,
                                                   int* __restrict__ rows, int B, int T, int E) {
    __shared__ int s_warp[8];
    __shared__ int s_base;
    const int g = blockIdx.x;
    const int t = g / E, e = g % E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_base = 0;
    __syncthreads();
    int* out = rows + offsets[g];
    for (int b0 = 0; b0 < B; b0 += 256) {
        const int b = b0 + threadIdx.x;
        const bool on = b < B && gates[((size_t)b * T + t) * E + e] > 0.f;
        const unsigned m = __ballot_sync(0xffffffffu, on);
        if (lane == 0) s_warp[warp] = __popc(m);
        __syncthreads();
        int before = s_base;
        for (int w = 0; w < warp; ++w) before += s_warp[w];
        if (on) out[before + __popc(m & ((1u << lane) - 1u))] = b;
        __syncthreads();
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int w = 0; w < 8; ++w) tot += s_warp[w];
            s_base += tot;
        }
        __syncthreads();
    }
}

// ---- 5: gather active rows ------------------------------------------------------------
template <typename Ein, typename Eout>
__global__ void gather_kernel(const Ein* __restrict__ S, long long s_sb, long long s_st,
                              const int* __restrict__ counts, const int* __restrict__ offsets,
                              const int* __restrict__ rows, Eout* __restrict__ Sg, int D, int NE) {
    const int g = blockIdx.y;
    const int t = g / NE;
    const int cnt = counts[g], off = offsets[g];
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int i = blockIdx.x * wpb + (threadIdx.x >> 5); i < cnt; i += gridDim.x * wpb) {
        const int b = rows[off + i];
        const Ein* src = S + b * s_sb + t * s_st;
        Eout* dst = Sg + (size_t)(off + i) * D;
        for (int j = lane; j < D; j += 32) dst[j] = from_f32<Eout>(to_f32(src[j]));
    }
}

// ---- 6/7 on CUDA cores (float32 path and shapes the tensor-core kernel does not tile) ----
constexpr int TM = 64, TN = 64, TK = 16;

// EPI 1: out[row][n] = Gelu(acc + b1) (activation dtype), rows packed;
// EPI 2: V[b, t] += gate (acc + b2).  Launch group j -> weight group base + j stride.
template <typename Tin, int EPI>
__global__ void __launch_bounds__(256)
moe_gemm_simt_kernel(const Tin* __restrict__ A, const Tin* __restrict__ W, const float* __restrict__ bias,
                     Tin* __restrict__ hout, const int* __restrict__ counts, const int* __restrict__ offsets,
                     const int* __restrict__ rows, const float* __restrict__ gates, float* __restrict__ V,
                     long long v_sb, long long v_st, int N, int K, int T, int NE, int base, int stride) {
    __shared__ float As[TK][TM + 4];
    __shared__ float Ws[TK][TN + 4];
    const int wg = base + blockIdx.z * stride;
    const int M = counts[wg];
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    if (m0 >= M) return;
    const long long row0 = offsets[wg];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const Tin* Ag = A + row0 * K;
    const Tin* Wt = W + (size_t)wg * N * K;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int lr = threadIdx.x >> 2;
    const int lk = (threadIdx.x & 3) * 4;
    for (int k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = k0 + lk + e;
            const int m = m0 + lr, n = n0 + lr;
            As[lk + e][lr] = (m < M && k < K) ? to_f32(Ag[(size_t)m * K + k]) : 0.f;
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
    const int t = wg / NE, ee = wg % NE;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= M) continue;
        if (EPI == 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx + 16 * j;
                if (n < N) hout[(size_t)(row0 + m) * N + n] = from_f32<Tin>(gelu_erf(acc[i][j] + bias[(size_t)wg * N + n]));
            }
        } else {
            const int b = rows[row0 + m];
            const float gate = gates[((size_t)b * T + t) * NE + ee];
            float* vrow = V + b * v_sb + t * v_st;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx + 16 * j;
                if (n < N) vrow[n] = fmaf(gate, acc[i][j] + bias[(size_t)wg * N + n], vrow[n]);
            }
        }
    }
}

template <typename Top>
__global__ void residual_z_kernel(const float* __restrict__ V, const Top* __restrict__ S, Top* __restrict__ Z, int B,
                                  int T, int D, int Bcap) {
    const long long n = (long long)T * B * D;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(i % D);
        const long long tb = i / D;
        const int b = (int)(tb % B), t = (int)(tb / B);
        const size_t o = ((size_t)t * Bcap + b) * D + j;
        Z[o] = from_f32<Top>(V[o] + to_f32(S[o]));
    }
}

template <typename T>
cudaError_t dalloc(T** p, size_t n, long long* bytes) {
    *p = nullptr;
    if (n == 0) return cudaSuccess;
    cudaError_t e = cudaMalloc((void**)p, n * sizeof(T));
    if (e != cudaSuccess) {
        *p = nullptr;
        return e;
    }
    if (bytes) *bytes += (long long)(n * sizeof(T));
    return cudaSuccess;
}

cudaError_t dalloc_bytes(void** p, size_t n, long long* bytes) {
    *p = nullptr;
    cudaError_t e = cudaMalloc(p, n);
    if (e != cudaSuccess) {
        *p = nullptr;
        return e;
    }
    if (bytes) *bytes += (long long)n;
    return cudaSuccess;
}

bool moe_use_tc(Act act, int D, int Fe) { return act == Act::BF16 && tc_supported(D, Fe); }

}  // namespace

cudaError_t moe_pack_weights(const MoeShape& ms, const void* Wg, const void* bg, const void* eW1, const void* eb1,
                             const void* eW2, const void* eb2, MoeWeights& w, long long* bytes, cudaStream_t s) {
    const size_t esz = op_size(ms.act);
    const size_t G = (size_t)ms.T * ms.E;
    cudaError_t e;
    if ((e = dalloc_bytes(&w.W1p, G * ms.Fe * ms.D * esz, bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&w.W2p, G * ms.D * ms.Fe * esz, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&w.b1, G * ms.Fe, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&w.b2, G * ms.D, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&w.Wg, (size_t)ms.T * ms.E * ms.D, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&w.bg, (size_t)ms.T * ms.E, bytes)) != cudaSuccess) return e;
    // eW1 [T][E][D][Fe] -> [T*E][Fe][D];  eW2 [T][E][Fe][D] -> [T*E][D][Fe]  (operand type)
    if ((e = launch_pack_transpose(ms.act, eW1, w.W1p, (int)G, ms.D, ms.Fe, s)) != cudaSuccess) return e;
    if ((e = launch_pack_transpose(ms.act, eW2, w.W2p, (int)G, ms.Fe, ms.D, s)) != cudaSuccess) return e;
    if ((e = launch_to_f32(ms.act, eb1, w.b1, G * ms.Fe, s)) != cudaSuccess) return e;
    if ((e = launch_to_f32(ms.act, eb2, w.b2, G * ms.D, s)) != cudaSuccess) return e;
    if ((e = launch_to_f32(ms.act, bg, w.bg, (size_t)ms.T * ms.E, s)) != cudaSuccess) return e;
    // Wg [T][D][E] -> float [T][D][E] -> [T][E][D]
    float* tmp = nullptr;
    if ((e = dalloc(&tmp, (size_t)ms.T * ms.D * ms.E, nullptr)) != cudaSuccess) return e;
    e = launch_to_f32(ms.act, Wg, tmp, (size_t)ms.T * ms.D * ms.E, s);
    if (e == cudaSuccess) e = launch_transpose_f32(tmp, w.Wg, ms.T, ms.D, ms.E, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(tmp);
    return e;
}

void moe_free_weights(MoeWeights& w) {
    cudaFree(w.W1p); cudaFree(w.W2p); cudaFree(w.b1); cudaFree(w.b2); cudaFree(w.Wg); cudaFree(w.bg);
    w = MoeWeights{};
}

cudaError_t moe_alloc_workspace(const MoeShape& ms, int Bcap, MoeWorkspace& ws, long long* bytes) {
    const size_t G = (size_t)ms.T * ms.E;
    const size_t esz = op_size(ms.act);
    ws.Bcap = Bcap;
    cudaError_t e;
    if ((e = dalloc(&ws.gates, (size_t)Bcap * G, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.counts, G, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.offsets, G + 1, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.rows, G * Bcap, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.tile_prefix, G + 1 + (size_t)ms.E * (ms.T + 1), bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&ws.Sg, G * Bcap * ms.D * esz, bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&ws.Hm, G * Bcap * ms.Fe * esz, bytes)) != cudaSuccess) return e;
    return cudaSuccess;
}

void moe_free_workspace(MoeWorkspace& ws) {
    cudaFree(ws.gates); cudaFree(ws.counts); cudaFree(ws.offsets); cudaFree(ws.rows); cudaFree(ws.tile_prefix);
    cudaFree(ws.pair_of_row); cudaFree(ws.Sg); cudaFree(ws.Hm);
    ws = MoeWorkspace{};
}

cudaError_t moe_forward(const MoeLaunch& ml, const MoeWeights& w, MoeWorkspace& ws, float* V, bool V_token_major,
                        float* gates_out, cudaStream_t s, const std::function<void*(int)>& prof_begin,
                        const std::function<void(void*)>& prof_end) {
    const int T = ml.T, D = ml.D, E = ml.E, Fe = ml.Fe, B = ml.B;
    const int G = T * E;
    const long long s_sb = ml.S_sample_major ? (long long)T * D : D;
    const long long s_st = ml.S_sample_major ? (long long)D : (long long)ml.Bcap * D;
    const long long v_sb = V_token_major ? D : (long long)T * D;
    const long long v_st = V_token_major ? (long long)ml.Bcap * D : D;
    const long long rows_cap = (long long)G * ws.Bcap;
    cudaError_t e;
    auto scoped = [&](int kind, auto&& fn) -> cudaError_t {
        void* h = prof_begin(kind);
        cudaError_t r = fn();
        prof_end(h);
        return r;
    };
    // 1-5: route, compact, gather
    e = scoped(6 /* RM_K_MOE_ROUTE */, [&]() -> cudaError_t {
        const long long warps = (long long)B * T;
        int grid = (int)((warps * 32 + 255) / 256);
        if (grid > ml.num_sms * 16) grid = ml.num_sms * 16;
        if (ml.act == Act::F32)
            router_kernel<float><<<grid, 256, 0, s>>>((const float*)ml.S, s_sb, s_st, w.Wg, w.bg, ws.gates, B, T, D, E);
        else if (ml.S_sample_major)   // the caller's bf16 S
            router_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)ml.S, s_sb, s_st, w.Wg, w.bg,
                                                               ws.gates, B, T, D, E);
        else                          // the stack's fp16 S
            router_kernel<__half><<<grid, 256, 0, s>>>((const __half*)ml.S, s_sb, s_st, w.Wg, w.bg, ws.gates, B, T, D,
                                                        E);
        count_kernel<<<G, 256, 0, s>>>(ws.gates, ws.counts, B, T, E);
        prefix_kernel<<<1, 32, 0, s>>>(ws.counts, ws.offsets, ws.tile_prefix, T, E);
        fill_kernel<<<G, 256, 0, s>>>(ws.gates, ws.offsets, ws.rows, B, T, E);
        dim3 gg((B + 7) / 8 < 64 ? (B + 7) / 8 : 64, G);
        if (ml.act == Act::F32)
            gather_kernel<float, float><<<gg, 256, 0, s>>>((const float*)ml.S, s_sb, s_st, ws.counts, ws.offsets,
                                                           ws.rows, (float*)ws.Sg, D, E);
        else if (ml.S_sample_major)
            gather_kernel<__nv_bfloat16, __half><<<gg, 256, 0, s>>>((const __nv_bfloat16*)ml.S, s_sb, s_st,
                                                                     ws.counts, ws.offsets, ws.rows, (__half*)ws.Sg,
                                                                     D, E);
        else
            gather_kernel<__half, __half><<<gg, 256, 0, s>>>((const __half*)ml.S, s_sb, s_st, ws.counts, ws.offsets,
                                                             ws.rows, (__half*)ws.Sg, D, E);
        if (gates_out) {
            cudaError_t r = cudaMemcpyAsync(gates_out, ws.gates, (size_t)B * G * sizeof(float),
                                            cudaMemcpyDeviceToDevice, s);
            if (r != cudaSuccess) return r;
        }
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    // V = 0 on the B rows of every token
    if (V_token_major)
        e = cudaMemset2DAsync(V, (size_t)ml.Bcap * D * sizeof(float), 0, (size_t)B * D * sizeof(float), T, s);
    else
        e = cudaMemsetAsync(V, 0, (size_t)B * T * D * sizeof(float), s);
    if (e != cudaSuccess) return e;

    const bool tc = moe_use_tc(ml.act, D, Fe);
    // 6: expert layer 1
    e = scoped(7 /* RM_K_MOE_GEMM1 */, [&]() -> cudaError_t {
        if (tc)
            return launch_moe_gemm1_tc(ws.Sg, rows_cap, w.W1p, w.b1, ws.Hm, G, D, Fe, ws.counts, ws.offsets,
                                       ws.tile_prefix, ml.num_sms, ml.err, kMoeWaitTimeoutNs, s);
        dim3 grid((Fe + TN - 1) / TN, (B + TM - 1) / TM, G);
        if (ml.act == Act::BF16)
            moe_gemm_simt_kernel<__half, 1><<<grid, 256, 0, s>>>((const __half*)ws.Sg, (const __half*)w.W1p, w.b1,
                                                                 (__half*)ws.Hm, ws.counts, ws.offsets, ws.rows,
                                                                 nullptr, nullptr, 0, 0, Fe, D, T, E, 0, 1);
        else
            moe_gemm_simt_kernel<float, 1><<<grid, 256, 0, s>>>((const float*)ws.Sg, (const float*)w.W1p, w.b1,
                                                                (float*)ws.Hm, ws.counts, ws.offsets, ws.rows, nullptr,
                                                                nullptr, 0, 0, Fe, D, T, E, 0, 1);
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    // 7: expert layer 2, gated accumulation, one launch per expert index
    for (int ei = 0; ei < E; ++ei) {
        e = scoped(8 /* RM_K_MOE_GEMM2 */, [&]() -> cudaError_t {
            const int* tp = ws.tile_prefix + G + 1 + ei * (T + 1);
            if (tc)
                return launch_moe_gemm2_tc(ws.Hm, rows_cap, w.W2p, w.b2, T, E, ei, D, Fe, ws.counts, ws.offsets, tp,
                                           ws.rows, ws.gates, V, v_sb, v_st, ml.num_sms, ml.err, kMoeWaitTimeoutNs,
                                           s);
            dim3 grid((D + TN - 1) / TN, (B + TM - 1) / TM, T);
            if (ml.act == Act::BF16)
                moe_gemm_simt_kernel<__half, 2><<<grid, 256, 0, s>>>((const __half*)ws.Hm, (const __half*)w.W2p, w.b2,
                                                                     nullptr, ws.counts, ws.offsets, ws.rows,
                                                                     ws.gates, V, v_sb, v_st, D, Fe, T, E, ei, E);
            else
                moe_gemm_simt_kernel<float, 2><<<grid, 256, 0, s>>>((const float*)ws.Hm, (const float*)w.W2p, w.b2,
                                                                    nullptr, ws.counts, ws.offsets, ws.rows, ws.gates,
                                                                    V, v_sb, v_st, D, Fe, T, E, ei, E);
            return cudaGetLastError();
        });
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t moe_residual_z(Act act, const float* V, const void* S, void* Z, int B, int T, int D, int Bcap,
                           cudaStream_t s) {
    const long long n = (long long)T * B * D;
    int grid = (int)((n + 255) / 256);
    if (grid > 152 * 16) grid = 152 * 16;
    if (act == Act::BF16)
        residual_z_kernel<__half><<<grid, 256, 0, s>>>(V, (const __half*)S, (__half*)Z, B, T, D, Bcap);
    else
        residual_z_kernel<float><<<grid, 256, 0, s>>>(V, (const float*)S, (float*)Z, B, T, D, Bcap);
    return cudaGetLastError();
}

}  // namespace rm
