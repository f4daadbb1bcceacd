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
//   1 route       one pass over S: G = ReLU(s Wg_t + bg_t); each open (b, t, e)
//                 claims a slot of group t E + e and copies s into it (fp16
//                 operands for bf16 contexts); V rows with no open expert are zeroed
//   2 tiles       128-row tile prefix sums per launch
//   3 expert L1   variable-size grouped GEMM + bias + GELU -> Hm (packed rows)
//   4 expert L2   one launch per expert index e (fixed order e = 0..E-1):
//                 V[b, t] (+)= G * (Hm W2_{t,e} + b2_{t,e}), the first open
//                 expert of (b, t) storing and the later ones adding
// The fixed order of step 4 makes the float32 sum over experts deterministic.
#include <type_traits>
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
                                const int* row_sample, const float* gates, const int* first_e, float* V,
                                long long v_sb, long long v_st, int num_sms, int* err, unsigned long long timeout_ns,
                                cudaStream_t s);

namespace {

constexpr unsigned long long kMoeWaitTimeoutNs = 2000000000ull;

// ---- 1: route (gates, slot claim, gather) ------------------------------------------
// One warp takes RQ = 4 samples of one token t at a time.  Each lane walks its
// columns of the 4 rows in chunks of CH elements (16-byte loads when the rows
// allow), and accumulates the 4 x 8 partial dot products with an 8-expert slice
// of Wg_t (fp32, read through L1: every warp of the CTA works on the same
// token).  A transpose-reduction (31 shuffles) leaves lane l holding the full
// sum for row l / 8 and expert l % 8 of the slice.  Each open (row, expert)
// claims a slot of its group g = t E + e by an atomic on counts[g]; the slot's
// packed row is g Bcap + slot, so the gathered rows of group g are the first
// counts[g] rows of its fixed Bcap-row block.  The warp then copies each open
// row into its slot, converted to the operand type.  A (sample, token) with
// no open expert gets its V row zeroed here (the expert layer-2 launches write
// the rows of the others; the first open expert stores, later ones add).
//
// The order of rows inside a group follows the atomics and may change from
// run to run; no value does: each output row's arithmetic is independent of
// its position in a tile, and the experts are combined in a fixed order.
constexpr int kRouteRows = 4;       // samples per warp pass
constexpr int kRouteExp = 8;        // experts per pass (kRouteRows * kRouteExp == 32)
constexpr int kRouteWarps = 8;
constexpr int kRouteSamplesPerCta = 128;

template <typename Tin, int CH>
__device__ __forceinline__ void load_chunk(const Tin* p, bool ok, float (&x)[CH]) {
    if constexpr (CH == 1) {
        x[0] = ok ? to_f32(p[0]) : 0.f;
    } else if constexpr (sizeof(Tin) == 4) {
        static_assert(CH == 4, "16-byte chunk of fp32");
        const float4 v = ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        static_assert(CH == 8, "16-byte chunk of 16-bit values");
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ok) v = __ldg(reinterpret_cast<const uint4*>(p));
        const Tin* h = reinterpret_cast<const Tin*>(&v);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = to_f32(h[k]);
    }
}

// CH consecutive floats (16-byte loads when CH is a multiple of 4)
template <int CH>
__device__ __forceinline__ void load_wf(const float* p, float (&w)[CH]) {
    if constexpr (CH % 4 == 0) {
#pragma unroll
        for (int q = 0; q < CH / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p) + q);
            w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < CH; ++k) w[k] = __ldg(p + k);
    }
}

template <typename Tin, typename Tout, int CH>
__device__ __forceinline__ void copy_row(const Tin* __restrict__ src, Tout* __restrict__ dst, int D, int lane) {
    for (int c0 = CH * lane; c0 < D; c0 += 32 * CH) {
        float x[CH];
        load_chunk<Tin, CH>(src + c0, true, x);
        if constexpr (CH == 8 && std::is_same_v<Tout, __half>) {
            uint4 o;
            uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = pack_f16x2(x[2 * k], x[2 * k + 1]);
            *reinterpret_cast<uint4*>(dst + c0) = o;
        } else if constexpr (CH == 4 && sizeof(Tout) == 4) {
            *reinterpret_cast<float4*>(dst + c0) = make_float4(x[0], x[1], x[2], x[3]);
        } else {
#pragma unroll
            for (int k = 0; k < CH; ++k) dst[c0 + k] = from_f32<Tout>(x[k]);
        }
    }
}

template <typename Tin, typename Tout, int CH>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const Tin* __restrict__ S, long long s_sb, long long s_st, const float* __restrict__ Wg,
             const float* __restrict__ bg, float* __restrict__ gates, int* __restrict__ counts,
             int* __restrict__ rows, int* __restrict__ first_e, Tout* __restrict__ Sg, float* __restrict__ V,
             long long v_sb, long long v_st, int B, int T, int D, int E, int Bcap) {
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int my_r = lane / kRouteExp, my_e = lane % kRouteExp;
    const int b_end = min(B, (int)(blockIdx.x + 1) * kRouteSamplesPerCta);
    for (int b0 = blockIdx.x * kRouteSamplesPerCta + warp * kRouteRows; b0 < b_end; b0 += kRouteWarps * kRouteRows) {
        const Tin* row[kRouteRows];
        bool ok[kRouteRows];
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r) {
            ok[r] = b0 + r < b_end;
            row[r] = S + (long long)(ok[r] ? b0 + r : b0) * s_sb + (long long)t * s_st;
        }
        int first = E;                               // first open expert of this lane's row (my_r)
        for (int e0 = 0; e0 < E; e0 += kRouteExp) {
            const int ne = min(kRouteExp, E - e0);
            float acc[kRouteRows * kRouteExp];
#pragma unroll
            for (int i = 0; i < kRouteRows * kRouteExp; ++i) acc[i] = 0.f;
            const float* wt = Wg + ((size_t)t * E + e0) * D;
            for (int c0 = CH * lane; c0 < D; c0 += 32 * CH) {
                float x[kRouteRows][CH];
#pragma unroll
                for (int r = 0; r < kRouteRows; ++r) load_chunk<Tin, CH>(row[r] + c0, ok[r], x[r]);
#pragma unroll
                for (int e = 0; e < kRouteExp; ++e) {
                    if (e < ne) {
                        float w[CH];
                        load_wf<CH>(wt + (size_t)e * D + c0, w);
#pragma unroll
                        for (int r = 0; r < kRouteRows; ++r)
#pragma unroll
                            for (int k = 0; k < CH; ++k) acc[r * kRouteExp + e] = fmaf(x[r][k], w[k], acc[r * kRouteExp + e]);
                    }
                }
            }
            // transpose-reduction: after the step with offset o, a lane keeps the half of
            // the remaining values selected by its bit o; lane l ends with value l's sum
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < o; ++i) {
                    const float send = upper ? acc[i] : acc[i + o];
                    const float keep = upper ? acc[i + o] : acc[i];
                    acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            const int b = b0 + my_r, e = e0 + my_e;
            const bool mine = my_e < ne && ok[my_r];
            const float g = mine ? fmaxf(acc[0] + __ldg(bg + (size_t)t * E + e), 0.f) : 0.f;
            if (mine) gates[((size_t)b * T + t) * E + e] = g;
            const bool open = mine && g > 0.f;
            int slot = 0;
            if (open) {
                const int grp = t * E + e;
                slot = atomicAdd(counts + grp, 1);
                rows[(size_t)grp * Bcap + slot] = b;
            }
            unsigned m = __ballot_sync(0xffffffffu, open);
            const unsigned row_bits = (m >> (my_r * kRouteExp)) & ((1u << kRouteExp) - 1u);
            if (first == E && row_bits) first = e0 + __ffs(row_bits) - 1;
            while (m) {
                const int l = __ffs(m) - 1;
                m &= m - 1;
                const int sl = __shfl_sync(0xffffffffu, slot, l);
                const int r = l / kRouteExp;
                const int grp = t * E + e0 + l % kRouteExp;
                copy_row<Tin, Tout, CH>(S + (long long)(b0 + r) * s_sb + (long long)t * s_st,
                                        Sg + ((size_t)grp * Bcap + sl) * D, D, lane);
            }
        }
        if (my_e == 0 && ok[my_r]) first_e[(size_t)(b0 + my_r) * T + t] = first;
        // V rows of samples with no open expert are zero
        const unsigned closed_rows = __ballot_sync(0xffffffffu, my_e == 0 && first == E);
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r) {
            if (ok[r] && (closed_rows >> (r * kRouteExp)) & 1u) {
                float* vrow = V + (long long)(b0 + r) * v_sb + (long long)t * v_st;
                for (int c = lane; c < D; c += 32) vrow[c] = 0.f;
            }
        }
    }
}

// ---- 2: tile prefixes -------------------------------------------------------------
// offsets[g] = g Bcap (fixed blocks); tile_prefix[0 .. G] over g = t E + e (expert
// layer 1); tile_prefix[G + 1 + e (T + 1) + t] over t for fixed e (layer 2, one
// launch per e).  One CTA, each thread a contiguous run of groups.
constexpr int kTilesThreads = 1024;

__global__ void __launch_bounds__(kTilesThreads)
tiles_kernel(const int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ tile_prefix, int T, int E,
             int Bcap) {
    __shared__ int part[kTilesThreads];
    const int G = T * E;
    const int per = (G + kTilesThreads - 1) / kTilesThreads;
    const int g0 = threadIdx.x * per, g1 = min(G, g0 + per);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += (counts[g] + 127) / 128;
    part[threadIdx.x] = sum;
    __syncthreads();
    // inclusive scan of the per-thread sums (Hillis-Steele)
    for (int o = 1; o < kTilesThreads; o <<= 1) {
        const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int run = part[threadIdx.x] - sum;
    for (int g = g0; g < g1; ++g) {
        offsets[g] = g * Bcap;
        tile_prefix[g] = run;
        run += (counts[g] + 127) / 128;
    }
    if (threadIdx.x == kTilesThreads - 1) {
        tile_prefix[G] = part[kTilesThreads - 1];
        offsets[G] = G * Bcap;
    }
    for (int e = threadIdx.x; e < E; e += kTilesThreads) {
        int* p = tile_prefix + G + 1 + e * (T + 1);
        int acc = 0;
        for (int t = 0; t < T; ++t) {
            p[t] = acc;
            acc += (counts[t * E + e] + 127) / 128;
        }
        p[T] = acc;
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
                     const int* __restrict__ rows, const float* __restrict__ gates, const int* __restrict__ first_e,
                     float* __restrict__ V,
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
            const bool first = first_e[(size_t)b * T + t] == ee;   // the first open expert stores
            float* vrow = V + b * v_sb + t * v_st;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx + 16 * j;
                if (n < N) vrow[n] = fmaf(gate, acc[i][j] + bias[(size_t)wg * N + n], first ? 0.f : vrow[n]);
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
    if ((e = dalloc(&ws.first_e, (size_t)Bcap * ms.T, bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&ws.Sg, G * Bcap * ms.D * esz, bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&ws.Hm, G * Bcap * ms.Fe * esz, bytes)) != cudaSuccess) return e;
    return cudaSuccess;
}

void moe_free_workspace(MoeWorkspace& ws) {
    cudaFree(ws.gates); cudaFree(ws.counts); cudaFree(ws.offsets); cudaFree(ws.rows); cudaFree(ws.tile_prefix);
    cudaFree(ws.first_e); cudaFree(ws.Sg); cudaFree(ws.Hm);
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
    // 1-2: route (gates, slots, gather, zero rows), tile prefixes
    e = scoped(6 /* RM_K_MOE_ROUTE */, [&]() -> cudaError_t {
        cudaError_t r = cudaMemsetAsync(ws.counts, 0, (size_t)G * sizeof(int), s);
        if (r != cudaSuccess) return r;
        const dim3 grid((B + kRouteSamplesPerCta - 1) / kRouteSamplesPerCta, T);
        const int esz = ml.act == Act::F32 ? 4 : 2;
        const bool vec = ((uintptr_t)ml.S % 16 == 0) && (D % (16 / esz) == 0) && (s_sb * esz % 16 == 0) &&
                         (s_st * esz % 16 == 0);
#define RM_ROUTE(TIN, TOUT, CH)                                                                               \
    route_kernel<TIN, TOUT, CH><<<grid, kRouteWarps * 32, 0, s>>>((const TIN*)ml.S, s_sb, s_st, w.Wg, w.bg,    \
                                                                   ws.gates, ws.counts, ws.rows, ws.first_e,   \
                                                                   (TOUT*)ws.Sg,                               \
                                                                   V, v_sb, v_st, B, T, D, E, ws.Bcap)
        if (ml.act == Act::F32) {
            if (vec) RM_ROUTE(float, float, 4); else RM_ROUTE(float, float, 1);
        } else if (ml.S_sample_major) {   // the caller's bf16 S
            if (vec) RM_ROUTE(__nv_bfloat16, __half, 8); else RM_ROUTE(__nv_bfloat16, __half, 1);
        } else {                          // the stack's fp16 S
            if (vec) RM_ROUTE(__half, __half, 8); else RM_ROUTE(__half, __half, 1);
        }
#undef RM_ROUTE
        tiles_kernel<<<1, kTilesThreads, 0, s>>>(ws.counts, ws.offsets, ws.tile_prefix, T, E, ws.Bcap);
        if (gates_out) {
            r = cudaMemcpyAsync(gates_out, ws.gates, (size_t)B * G * sizeof(float), cudaMemcpyDeviceToDevice, s);
            if (r != cudaSuccess) return r;
        }
        return cudaGetLastError();
    });
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
                                                                 nullptr, nullptr, nullptr, 0, 0, Fe, D, T, E, 0, 1);
        else
            moe_gemm_simt_kernel<float, 1><<<grid, 256, 0, s>>>((const float*)ws.Sg, (const float*)w.W1p, w.b1,
                                                                (float*)ws.Hm, ws.counts, ws.offsets, ws.rows, nullptr,
                                                                nullptr, nullptr, 0, 0, Fe, D, T, E, 0, 1);
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    // 7: expert layer 2, gated accumulation, one launch per expert index
    for (int ei = 0; ei < E; ++ei) {
        e = scoped(8 /* RM_K_MOE_GEMM2 */, [&]() -> cudaError_t {
            const int* tp = ws.tile_prefix + G + 1 + ei * (T + 1);
            if (tc)
                return launch_moe_gemm2_tc(ws.Hm, rows_cap, w.W2p, w.b2, T, E, ei, D, Fe, ws.counts, ws.offsets, tp,
                                           ws.rows, ws.gates, ws.first_e, V, v_sb, v_st, ml.num_sms, ml.err,
                                           kMoeWaitTimeoutNs, s);
            dim3 grid((D + TN - 1) / TN, (B + TM - 1) / TM, T);
            if (ml.act == Act::BF16)
                moe_gemm_simt_kernel<__half, 2><<<grid, 256, 0, s>>>((const __half*)ws.Hm, (const __half*)w.W2p, w.b2,
                                                                     nullptr, ws.counts, ws.offsets, ws.rows,
                                                                     ws.gates, ws.first_e, V, v_sb, v_st, D, Fe, T, E,
                                                                     ei, E);
            else
                moe_gemm_simt_kernel<float, 2><<<grid, 256, 0, s>>>((const float*)ws.Hm, (const float*)w.W2p, w.b2,
                                                                    nullptr, ws.counts, ws.offsets, ws.rows, ws.gates,
                                                                    ws.first_e, V, v_sb, v_st, D, Fe, T, E, ei, E);
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
