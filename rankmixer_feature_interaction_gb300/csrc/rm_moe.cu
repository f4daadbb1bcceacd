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
//                 operands for bf16 contexts)
//   2 tiles       128-row tile prefix sums over the groups
//   3 expert L1   variable-size grouped GEMM + bias + GELU -> Hm (packed rows)
//   4 expert L2   the same over all groups, + bias, times the row's gate -> Y
//                 (packed rows, written over the gathered rows)
//   5 combine     V[b, t] = sum of the open experts' Y rows in ascending e
// The fixed order of step 5 makes the float32 sum over experts deterministic.
#include <type_traits>
#include <vector>

#include "rm_common.cuh"
#include "rm_internal.h"
#include "rm_moe.h"

namespace rm {

// tcgen05 launchers (rm_gemm_tc.cu)
cudaError_t launch_moe_gemm1_tc(const void* Sg, long long rows_total, const void* W1p, const float* b1, void* Hm,
                                int groups, int D, int Fe, const int* g_count, const int* g_off,
                                const int* tile_prefix, const int* tile_prefix256, int num_sms, int* err,
                                unsigned long long timeout_ns, cudaStream_t s);
cudaError_t launch_moe_gemm2_tc(const void* Hm, long long rows_total, const void* W2p, const float* b2, void* Y,
                                int groups, int D, int Fe, const int* g_count, const int* g_off,
                                const int* tile_prefix, const int* tile_prefix256, const float* row_gate,
                                int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s);

namespace {

constexpr unsigned long long kMoeWaitTimeoutNs = 2000000000ull;
constexpr int kMoePairMinBatch = 512;

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
// row into its slot, converted to the operand type, and records the slot
// (slot_of[b][t][e], -1 when closed) and the gate of the packed row.
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

// 8 16-bit values (bf16 or fp16) of a 16-byte chunk -> float
template <typename Tin>
__device__ __forceinline__ void to_f32x8_any(const uint4 v, float (&x)[8]) {
    const Tin* h = reinterpret_cast<const Tin*>(&v);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = to_f32(h[k]);
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
             float* __restrict__ row_gate, int* __restrict__ slot_of, Tout* __restrict__ Sg, int B, int T, int D,
             int E, int Bcap) {
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
            int slot = -1;
            if (open) {
                const int grp = t * E + e;
                slot = atomicAdd(counts + grp, 1);
                row_gate[(size_t)grp * Bcap + slot] = g;
            }
            if (mine) slot_of[((size_t)b * T + t) * E + e] = slot;      // -1: closed
            unsigned m = __ballot_sync(0xffffffffu, open);
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
    }
}

// Register-resident variant for 16-bit S with D = 256 NCH (NCH <= 8) and E <= 8
// (one expert slice): a warp takes 2 samples of token t per pass and holds
// both rows in registers (NCH 16-byte chunks per lane each), so the copies into
// the expert groups are stores only.  The 2 x 8 dot products reduce in 16
// shuffles; lane l then holds the sum for row (l >> 4) & 1, expert (l >> 1) & 7
// (lanes 2v and 2v + 1 hold the same value; the even one acts).
constexpr int kRoute2Rows = 2;

template <typename Tin, int NCH>
__global__ void __launch_bounds__(kRouteWarps * 32, 2)
route2_kernel(const Tin* __restrict__ S, long long s_sb, long long s_st, const float* __restrict__ Wg,
              const float* __restrict__ bg, float* __restrict__ gates, int* __restrict__ counts,
              float* __restrict__ row_gate, int* __restrict__ slot_of, __half* __restrict__ Sg, int B, int T,
              int D, int E, int Bcap) {
    static_assert(sizeof(Tin) == 2, "16-bit rows");
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int my_r = (lane >> 4) & 1, my_e = (lane >> 1) & 7;
    const bool lead = (lane & 1) == 0;
    const int b_end = min(B, (int)(blockIdx.x + 1) * kRouteSamplesPerCta);
    for (int b0 = blockIdx.x * kRouteSamplesPerCta + warp * kRoute2Rows; b0 < b_end;
         b0 += kRouteWarps * kRoute2Rows) {
        const bool ok0 = b0 < b_end, ok1 = b0 + 1 < b_end;
        const Tin* row0 = S + (long long)b0 * s_sb + (long long)t * s_st;
        const Tin* row1 = S + (long long)(ok1 ? b0 + 1 : b0) * s_sb + (long long)t * s_st;
        uint4 h0[NCH], h1[NCH];              // the rows: raw, then fp16
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            h0[i] = __ldg(reinterpret_cast<const uint4*>(row0 + 8 * lane + 256 * i));
            h1[i] = ok1 ? __ldg(reinterpret_cast<const uint4*>(row1 + 8 * lane + 256 * i)) : make_uint4(0u, 0u, 0u, 0u);
        }
        {
            const int e0 = 0, ne = E;
            float acc[2 * kRouteExp];
#pragma unroll
            for (int i = 0; i < 2 * kRouteExp; ++i) acc[i] = 0.f;
            const float* wt = Wg + ((size_t)t * E + e0) * D + 8 * lane;
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                float x0[8], x1[8];
                to_f32x8_any<Tin>(h0[i], x0);
                to_f32x8_any<Tin>(h1[i], x1);
#pragma unroll
                for (int e = 0; e < kRouteExp; ++e) {
                    if (e < ne) {
                        float w[8];
                        load_wf<8>(wt + (size_t)e * D + 256 * i, w);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            acc[e] = fmaf(x0[k], w[k], acc[e]);
                            acc[kRouteExp + e] = fmaf(x1[k], w[k], acc[kRouteExp + e]);
                        }
                    }
                }
                if (!std::is_same_v<Tin, __half>) {     // the chunk to fp16 for the copies
                    h0[i] = make_uint4(pack_f16x2(x0[0], x0[1]), pack_f16x2(x0[2], x0[3]), pack_f16x2(x0[4], x0[5]),
                                       pack_f16x2(x0[6], x0[7]));
                    h1[i] = make_uint4(pack_f16x2(x1[0], x1[1]), pack_f16x2(x1[2], x1[3]), pack_f16x2(x1[4], x1[5]),
                                       pack_f16x2(x1[6], x1[7]));
                }
            }
            // 16 values: halve by lane bits 4, 3, 2, 1, then add the pair (bit 0)
#pragma unroll
            for (int o = 16; o >= 2; o >>= 1) {
                const bool upper = (lane & o) != 0;
                const int half = o / 2;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = upper ? acc[i] : acc[i + half];
                    const float keep = upper ? acc[i + half] : acc[i];
                    acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
            const int b = b0 + my_r, e = e0 + my_e;
            const bool mine = lead && my_e < ne && (my_r == 0 ? ok0 : ok1);
            const float g = mine ? fmaxf(acc[0] + __ldg(bg + (size_t)t * E + e), 0.f) : 0.f;
            if (mine) gates[((size_t)b * T + t) * E + e] = g;
            const bool open = mine && g > 0.f;
            int slot = -1;
            if (open) {
                const int grp = t * E + e;
                slot = atomicAdd(counts + grp, 1);
                row_gate[(size_t)grp * Bcap + slot] = g;
            }
            if (mine) slot_of[((size_t)b * T + t) * E + e] = slot;
            unsigned m = __ballot_sync(0xffffffffu, open);
            while (m) {
                const int l = __ffs(m) - 1;
                m &= m - 1;
                const int sl = __shfl_sync(0xffffffffu, slot, l);
                const int grp = t * E + e0 + ((l >> 1) & 7);
                __half* dst = Sg + ((size_t)grp * Bcap + sl) * D + 8 * lane;
                if (((l >> 4) & 1) == 0) {
#pragma unroll
                    for (int i = 0; i < NCH; ++i) *reinterpret_cast<uint4*>(dst + 256 * i) = h0[i];
                } else {
#pragma unroll
                    for (int i = 0; i < NCH; ++i) *reinterpret_cast<uint4*>(dst + 256 * i) = h1[i];
                }
            }
        }
    }
}

// ---- 1b: route on the tensor cores -----------------------------------------------
// For 16-bit S, E <= 8 and D % 32 == 0: a warp takes 16 samples of token t and
// forms their 16 x E gate pre-activations as one chain of m16n8k16 MMAs over
// D (fp32 accumulation), instead of per-lane dot products that re-read Wg_t
// for every pair of rows.  Wg_t (fp32) enters as two fp16 parts, hi = fp16(w)
// and lo = fp16(w - hi), both multiplied in, so the weights keep about 21
// significant bits; S is exact in fp16 (bf16 LayerNorm outputs; values below
// fp16's normal range lose bits below 6e-8).  K is permuted inside each
// 32-column group so that a lane reads its rows as one 16-byte word per group:
// lane (g, c) holds columns 32 q + 8 c .. + 7 of rows g and g + 8, and k-step
// 2 q + h takes columns 32 q + 8 c + 4 h + {0, 1} into fragment slots a0 / a1
// and + {2, 3} into a2 / a3; the B fragments (precomputed per CTA in shared
// memory, hi and lo) follow the same map, so each gate sums the same products.
// Then the gates, slot claims and copies as in route_kernel; the copies re-read
// the open rows (from L2), a 16-byte word per lane.
constexpr int kRouteMmaWarps = 8;
constexpr int kRouteMmaTiles = 2;                                        // 16-sample tiles per warp
constexpr int kRouteMmaSamples = kRouteMmaWarps * kRouteMmaTiles * 16;   // per CTA

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two packed 16-bit inputs -> a packed fp16 pair (exact for bf16 values in fp16's range).
template <typename Tin> __device__ __forceinline__ uint32_t route_f16x2(uint32_t v);
template <> __device__ __forceinline__ uint32_t route_f16x2<__half>(uint32_t v) { return v; }
template <> __device__ __forceinline__ uint32_t route_f16x2<__nv_bfloat16>(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
template <typename Tin>
__device__ __forceinline__ uint4 route_f16x8(uint4 v) {
    return make_uint4(route_f16x2<Tin>(v.x), route_f16x2<Tin>(v.y), route_f16x2<Tin>(v.z), route_f16x2<Tin>(v.w));
}

size_t route_mma_smem(int D) { return (size_t)(D / 16) * 32 * sizeof(uint4); }

template <typename Tin>
__global__ void __launch_bounds__(kRouteMmaWarps * 32)
route_mma_kernel(const Tin* __restrict__ S, long long s_sb, long long s_st, const float* __restrict__ Wg,
                 const float* __restrict__ bg, float* __restrict__ gates, int* __restrict__ counts,
                 float* __restrict__ row_gate, int* __restrict__ slot_of, __half* __restrict__ Sg, int B, int T,
                 int D, int E, int Bcap) {
    extern __shared__ uint4 s_frag[];                 // [D / 16 k-steps][32 lanes]: b0, b1 hi; b0, b1 lo
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int nks = D >> 4, nq = D >> 5;
    for (int i = threadIdx.x; i < nks * 32; i += blockDim.x) {
        const int ks = i >> 5, ln = i & 31;
        const int gg = ln >> 2, cc = ln & 3;
        const int d0 = 32 * (ks >> 1) + 8 * cc + 4 * (ks & 1);     // physical columns d0 .. d0 + 3
        float w[4] = {0.f, 0.f, 0.f, 0.f};
        if (gg < E) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(Wg + ((size_t)t * E + gg) * D + d0));
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        }
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const __half h0 = __float2half_rn(w[2 * p]), h1 = __float2half_rn(w[2 * p + 1]);
            const __half l0 = __float2half_rn(w[2 * p] - __half2float(h0));
            const __half l1 = __float2half_rn(w[2 * p + 1] - __half2float(h1));
            hi[p] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            lo[p] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
        }
        s_frag[i] = make_uint4(hi[0], hi[1], lo[0], lo[1]);
    }
    __syncthreads();
    pdl_wait();              // S comes from the previous kernel of the stream
    pdl_launch_next();

    for (int tile = 0; tile < kRouteMmaTiles; ++tile) {
        const int b0 = blockIdx.x * kRouteMmaSamples + (warp * kRouteMmaTiles + tile) * 16;
        if (b0 >= B) break;
        const int r0 = b0 + g, r1 = b0 + g + 8;
        const bool ok0 = r0 < B, ok1 = r1 < B;
        const Tin* x0 = S + (long long)(ok0 ? r0 : b0) * s_sb + (long long)t * s_st + 8 * c;
        const Tin* x1 = S + (long long)(ok1 ? r1 : b0) * s_sb + (long long)t * s_st + 8 * c;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int q0 = 0; q0 < nq; q0 += 4) {
            uint4 v0[4], v1[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool in = q0 + u < nq;
                v0[u] = (in && ok0) ? __ldg(reinterpret_cast<const uint4*>(x0 + 32 * (q0 + u))) : make_uint4(0u, 0u, 0u, 0u);
                v1[u] = (in && ok1) ? __ldg(reinterpret_cast<const uint4*>(x1 + 32 * (q0 + u))) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (q0 + u < nq) {
                    const uint4 h0 = route_f16x8<Tin>(v0[u]), h1 = route_f16x8<Tin>(v1[u]);
                    const uint4 f0 = s_frag[(2 * (q0 + u)) * 32 + lane];
                    const uint4 f1 = s_frag[(2 * (q0 + u) + 1) * 32 + lane];
                    const uint32_t a0[4] = {h0.x, h1.x, h0.y, h1.y};
                    const uint32_t a1[4] = {h0.z, h1.z, h0.w, h1.w};
                    mma_f16_16816(acc, a0, f0.x, f0.y);
                    mma_f16_16816(acc, a0, f0.z, f0.w);
                    mma_f16_16816(acc, a1, f1.x, f1.y);
                    mma_f16_16816(acc, a1, f1.z, f1.w);
                }
            }
        }
        // lane (g, c): acc[0], acc[1] = row g, experts 2c, 2c + 1; acc[2], acc[3] = row g + 8
        int slot[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = (j < 2 ? r0 : r1), e = 2 * c + (j & 1);
            const bool mine = e < E && (j < 2 ? ok0 : ok1);
            const float gt = mine ? fmaxf(acc[j] + __ldg(bg + (size_t)t * E + e), 0.f) : 0.f;
            if (mine) gates[((size_t)row * T + t) * E + e] = gt;
            slot[j] = -1;
            if (mine && gt > 0.f) {
                const int grp = t * E + e;
                slot[j] = atomicAdd(counts + grp, 1);
                row_gate[(size_t)grp * Bcap + slot[j]] = gt;
            }
            if (mine) slot_of[((size_t)row * T + t) * E + e] = slot[j];
        }
        // the copies: one open (row, expert) at a time, the whole warp on its row
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            unsigned m = __ballot_sync(0xffffffffu, slot[j] >= 0);
            while (m) {
                const int l = __ffs(m) - 1;
                m &= m - 1;
                const int sl = __shfl_sync(0xffffffffu, slot[j], l);
                const int row = b0 + (l >> 2) + (j < 2 ? 0 : 8);
                const int grp = t * E + 2 * (l & 3) + (j & 1);
                const Tin* src = S + (long long)row * s_sb + (long long)t * s_st;
                __half* dst = Sg + ((size_t)grp * Bcap + sl) * D;
                // up to 8 16-byte words per lane in flight before any is stored; the
                // gathered rows are stored with the streaming hint, so that they do not
                // push out of L2 the S rows still to be re-read for the copies
                for (int k0 = 8 * lane; k0 < D; k0 += 2048) {
                    uint4 w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (k0 + 256 * i < D) w[i] = __ldg(reinterpret_cast<const uint4*>(src + k0 + 256 * i));
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (k0 + 256 * i < D) __stcs(reinterpret_cast<uint4*>(dst + k0 + 256 * i), route_f16x8<Tin>(w[i]));
                }
            }
        }
    }
}

// RM_MOE_ROUTE=dot in the environment keeps the per-lane dot-product router (a
// tuning switch: gates equal to float32 rounding, the same experts open).
bool route_mma_enabled() {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_MOE_ROUTE");
        env = (v && v[0] == 'd') ? 0 : 1;
    }
    return env == 1;
}

// ---- 2: tile prefixes -------------------------------------------------------------
// offsets[g] = g Bcap (fixed blocks); tile_prefix[0 .. G] over g = t E + e, the
// exclusive prefix of 128-row tiles (both expert layers tile their packed rows
// alike), and tile_prefix256 the same over 256-row tiles (CTA-pair tiles).
// One CTA, each thread a contiguous run of groups.
constexpr int kTilesThreads = 1024;

__global__ void __launch_bounds__(kTilesThreads)
tiles_kernel(const int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ tile_prefix,
             int* __restrict__ tile_prefix256, int T, int E, int Bcap) {
    __shared__ int part[2][kTilesThreads];
    const int G = T * E;
    const int per = (G + kTilesThreads - 1) / kTilesThreads;
    const int g0 = threadIdx.x * per, g1 = min(G, g0 + per);
    int sum = 0, sum2 = 0;
    for (int g = g0; g < g1; ++g) {
        sum += (counts[g] + 127) / 128;
        sum2 += (counts[g] + 255) / 256;
    }
    part[0][threadIdx.x] = sum;
    part[1][threadIdx.x] = sum2;
    __syncthreads();
    // inclusive scans of the per-thread sums (Hillis-Steele)
    for (int o = 1; o < kTilesThreads; o <<= 1) {
        const int v = threadIdx.x >= o ? part[0][threadIdx.x - o] : 0;
        const int v2 = threadIdx.x >= o ? part[1][threadIdx.x - o] : 0;
        __syncthreads();
        part[0][threadIdx.x] += v;
        part[1][threadIdx.x] += v2;
        __syncthreads();
    }
    int run = part[0][threadIdx.x] - sum, run2 = part[1][threadIdx.x] - sum2;
    for (int g = g0; g < g1; ++g) {
        offsets[g] = g * Bcap;
        tile_prefix[g] = run;
        tile_prefix256[g] = run2;
        run += (counts[g] + 127) / 128;
        run2 += (counts[g] + 255) / 256;
    }
    if (threadIdx.x == kTilesThreads - 1) {
        tile_prefix[G] = part[0][kTilesThreads - 1];
        tile_prefix256[G] = part[1][kTilesThreads - 1];
        offsets[G] = G * Bcap;
    }
}

// ---- 6/7 on CUDA cores (float32 path and shapes the tensor-core kernel does not tile) ----
constexpr int TM = 64, TN = 64, TK = 16;

// Packed rows of group wg = blockIdx.z, out in the operand type, same row index as A:
// EPI 1: out[row][n] = Gelu(acc + b1);  EPI 2: out[row][n] = row_gate[row] (acc + b2).
template <typename Tin, int EPI>
__global__ void __launch_bounds__(256)
moe_gemm_simt_kernel(const Tin* __restrict__ A, const Tin* __restrict__ W, const float* __restrict__ bias,
                     Tin* __restrict__ hout, const int* __restrict__ counts, const int* __restrict__ offsets,
                     const float* __restrict__ row_gate, int N, int K) {
    __shared__ float As[TK][TM + 4];
    __shared__ float Ws[TK][TN + 4];
    const int wg = blockIdx.z;
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
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= M) continue;
        const float gate = EPI == 2 ? row_gate[row0 + m] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n >= N) continue;
            const float u = acc[i][j] + bias[(size_t)wg * N + n];
            hout[(size_t)(row0 + m) * N + n] = from_f32<Tin>(EPI == 1 ? gelu_erf(u) : gate * u);
        }
    }
}

// ---- 5b: combine, 16-bit rows held whole -------------------------------------------------
// The same sums for fp16 rows with D % 256 == 0 and D <= 8 * 256: a lane loads
// all its 8-column words of one open expert's row before adding any (up to 8
// 16-byte loads in flight instead of one), then the next expert, ascending e,
// so every element is summed in the same order as in combine_kernel.
template <int NCH>
__global__ void __launch_bounds__(256)
combine_rows_kernel(const __half* __restrict__ Y, const int* __restrict__ slot_of, float* __restrict__ V,
                    long long v_sb, long long v_st, int B, int T, int D, int E, int Bcap) {
    const int lane = threadIdx.x & 31;
    const long long w0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = w0; r < (long long)B * T; r += nw) {
        const int b = (int)(r / T), t = (int)(r % T);
        const int* so = slot_of + r * E;
        float* vrow = V + (long long)b * v_sb + (long long)t * v_st;
        float acc[NCH][8];
#pragma unroll
        for (int i = 0; i < NCH; ++i)
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[i][k] = 0.f;
        for (int e = 0; e < E; ++e) {
            const int sl = __ldg(so + e);
            if (sl < 0) continue;
            const __half* y = Y + ((size_t)(t * E + e) * Bcap + sl) * D + 8 * lane;
            uint4 w[NCH];
#pragma unroll
            for (int i = 0; i < NCH; ++i)
                if (256 * i < D) w[i] = __ldg(reinterpret_cast<const uint4*>(y + 256 * i));
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                if (256 * i < D) {
                    const __half2* h = reinterpret_cast<const __half2*>(&w[i]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 f = __half22float2(h[q]);
                        acc[i][2 * q] += f.x;
                        acc[i][2 * q + 1] += f.y;
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            if (256 * i < D) {
                float4* dst = reinterpret_cast<float4*>(vrow + 8 * lane + 256 * i);
                dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
                dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
            }
        }
    }
}

// ---- 5: combine -----------------------------------------------------------------------
// V[b, t] = sum over the open experts e of (b, t), ascending, of their gated rows
// Y[slot_of[b][t][e] of group t E + e] (zero when none is open).  One warp per
// (b, t); each lane sums CH-column chunks in float32.
template <typename Ty, int CH>
__global__ void __launch_bounds__(256)
combine_kernel(const Ty* __restrict__ Y, const int* __restrict__ slot_of, float* __restrict__ V, long long v_sb,
               long long v_st, int B, int T, int D, int E, int Bcap) {
    const int lane = threadIdx.x & 31;
    const long long w0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = w0; r < (long long)B * T; r += nw) {
        const int b = (int)(r / T), t = (int)(r % T);
        const int* so = slot_of + r * E;
        float* vrow = V + (long long)b * v_sb + (long long)t * v_st;
        for (int c0 = CH * lane; c0 < D; c0 += 32 * CH) {
            float acc[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k) acc[k] = 0.f;
            for (int e = 0; e < E; ++e) {
                const int sl = __ldg(so + e);
                if (sl < 0) continue;
                float y[CH];
                load_chunk<Ty, CH>(Y + ((size_t)(t * E + e) * Bcap + sl) * D + c0, true, y);
#pragma unroll
                for (int k = 0; k < CH; ++k) acc[k] += y[k];
            }
            if constexpr (CH % 4 == 0) {
#pragma unroll
                for (int q = 0; q < CH / 4; ++q)
                    reinterpret_cast<float4*>(vrow + c0)[q] =
                        make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
            } else {
#pragma unroll
                for (int k = 0; k < CH; ++k) vrow[c0 + k] = acc[k];
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
    cudaError_t e = device_alloc((void**)p, n * sizeof(T));
    if (e != cudaSuccess) {
        *p = nullptr;
        return e;
    }
    if (bytes) *bytes += (long long)(n * sizeof(T));
    return cudaSuccess;
}

cudaError_t dalloc_bytes(void** p, size_t n, long long* bytes) {
    *p = nullptr;
    cudaError_t e = device_alloc(p, n);
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
    device_free(tmp);
    return e;
}

cudaError_t moe_pack_router(const MoeShape& ms, const void* Wg, const void* bg, float** Wg_out, float** bg_out,
                            long long* bytes, cudaStream_t s) {
    cudaError_t e;
    if ((e = dalloc(Wg_out, (size_t)ms.T * ms.E * ms.D, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(bg_out, (size_t)ms.T * ms.E, bytes)) != cudaSuccess) return e;
    if ((e = launch_to_f32(ms.act, bg, *bg_out, (size_t)ms.T * ms.E, s)) != cudaSuccess) return e;
    float* tmp = nullptr;
    if ((e = dalloc(&tmp, (size_t)ms.T * ms.D * ms.E, nullptr)) != cudaSuccess) return e;
    e = launch_to_f32(ms.act, Wg, tmp, (size_t)ms.T * ms.D * ms.E, s);
    if (e == cudaSuccess) e = launch_transpose_f32(tmp, *Wg_out, ms.T, ms.D, ms.E, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    device_free(tmp);
    return e;
}

void moe_free_weights(MoeWeights& w) {
    device_free(w.W1p); device_free(w.W2p); device_free(w.b1); device_free(w.b2); device_free(w.Wg); device_free(w.bg);
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
    if ((e = dalloc(&ws.row_gate, G * Bcap, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.slot_of, (size_t)Bcap * G, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.tile_prefix, G + 1, bytes)) != cudaSuccess) return e;
    if ((e = dalloc(&ws.tile_prefix256, G + 1, bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&ws.Sg, G * Bcap * ms.D * esz, bytes)) != cudaSuccess) return e;
    if ((e = dalloc_bytes(&ws.Hm, G * Bcap * ms.Fe * esz, bytes)) != cudaSuccess) return e;
    return cudaSuccess;
}

void moe_free_workspace(MoeWorkspace& ws) {
    device_free(ws.gates); device_free(ws.counts); device_free(ws.offsets); device_free(ws.row_gate); device_free(ws.slot_of);
    device_free(ws.tile_prefix); device_free(ws.tile_prefix256); device_free(ws.Sg); device_free(ws.Hm);
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
    // 1-2: route (gates, slots, gather), tile prefixes
    e = scoped(6 /* RM_K_MOE_ROUTE */, [&]() -> cudaError_t {
        cudaError_t r = cudaMemsetAsync(ws.counts, 0, (size_t)G * sizeof(int), s);
        if (r != cudaSuccess) return r;
        const dim3 grid((B + kRouteSamplesPerCta - 1) / kRouteSamplesPerCta, T);
        const int esz = ml.act == Act::F32 ? 4 : 2;
        const bool vec = ((uintptr_t)ml.S % 16 == 0) && (D % (16 / esz) == 0) && (s_sb * esz % 16 == 0) &&
                         (s_st * esz % 16 == 0);
#define RM_ROUTE(TIN, TOUT, CH)                                                                               \
    route_kernel<TIN, TOUT, CH><<<grid, kRouteWarps * 32, 0, s>>>((const TIN*)ml.S, s_sb, s_st, w.Wg, w.bg,    \
                                                                   ws.gates, ws.counts, ws.row_gate,           \
                                                                   ws.slot_of, (TOUT*)ws.Sg, B, T, D, E, ws.Bcap)
        const int nch = D / 256;
        const bool regs = ml.act != Act::F32 && vec && E <= kRouteExp && D % 256 == 0 && nch >= 1 && nch <= 8;
#define RM_ROUTE2(TIN, NCH)                                                                                  \
    route2_kernel<TIN, NCH><<<grid, kRouteWarps * 32, 0, s>>>((const TIN*)ml.S, s_sb, s_st, w.Wg, w.bg, ws.gates, \
                                                              ws.counts, ws.row_gate, ws.slot_of, (__half*)ws.Sg,  \
                                                              B, T, D, E, ws.Bcap)
#define RM_ROUTE2_N(TIN)                                                                                     \
    switch (nch) {                                                                                           \
        case 1: RM_ROUTE2(TIN, 1); break;                                                                    \
        case 2: RM_ROUTE2(TIN, 2); break;                                                                    \
        case 3: RM_ROUTE2(TIN, 3); break;                                                                    \
        case 4: RM_ROUTE2(TIN, 4); break;                                                                    \
        case 5: RM_ROUTE2(TIN, 5); break;                                                                    \
        case 6: RM_ROUTE2(TIN, 6); break;                                                                    \
        case 7: RM_ROUTE2(TIN, 7); break;                                                                    \
        default: RM_ROUTE2(TIN, 8); break;                                                                   \
    }
        const bool mma = ml.act != Act::F32 && vec && E <= 8 && D % 32 == 0 && route_mma_enabled() &&
                         route_mma_smem(D) <= 96 * 1024;
        const dim3 mgrid((B + kRouteMmaSamples - 1) / kRouteMmaSamples, T);
        if (mma) {
            const size_t smem = route_mma_smem(D);
            cudaError_t ee;
            if (ml.S_sample_major) {
                ee = cudaFuncSetAttribute(route_mma_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
                if (ee != cudaSuccess) return ee;
                launch_k(route_mma_kernel<__nv_bfloat16>, mgrid, dim3(kRouteMmaWarps * 32), smem, s,
                         (const __nv_bfloat16*)ml.S, s_sb, s_st, (const float*)w.Wg, (const float*)w.bg, ws.gates,
                         ws.counts, ws.row_gate, ws.slot_of, (__half*)ws.Sg, B, T, D, E, ws.Bcap);
            } else {
                ee = cudaFuncSetAttribute(route_mma_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
                if (ee != cudaSuccess) return ee;
                launch_k(route_mma_kernel<__half>, mgrid, dim3(kRouteMmaWarps * 32), smem, s, (const __half*)ml.S,
                         s_sb, s_st, (const float*)w.Wg, (const float*)w.bg, ws.gates, ws.counts, ws.row_gate,
                         ws.slot_of, (__half*)ws.Sg, B, T, D, E, ws.Bcap);
            }
        } else if (ml.act == Act::F32) {
            if (vec) RM_ROUTE(float, float, 4); else RM_ROUTE(float, float, 1);
        } else if (ml.S_sample_major) {   // the caller's bf16 S
            if (regs) { RM_ROUTE2_N(__nv_bfloat16) }
            else if (vec) RM_ROUTE(__nv_bfloat16, __half, 8);
            else RM_ROUTE(__nv_bfloat16, __half, 1);
        } else {                          // the stack's fp16 S
            if (regs) { RM_ROUTE2_N(__half) }
            else if (vec) RM_ROUTE(__half, __half, 8);
            else RM_ROUTE(__half, __half, 1);
        }
#undef RM_ROUTE2_N
#undef RM_ROUTE2
#undef RM_ROUTE
        tiles_kernel<<<1, kTilesThreads, 0, s>>>(ws.counts, ws.offsets, ws.tile_prefix, ws.tile_prefix256, T, E,
                                                 ws.Bcap);
        if (gates_out) {
            r = cudaMemcpyAsync(gates_out, ws.gates, (size_t)B * G * sizeof(float), cudaMemcpyDeviceToDevice, s);
            if (r != cudaSuccess) return r;
        }
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    const bool tc = moe_use_tc(ml.act, D, Fe);
    // CTA-pair tiles (256 rows) when the groups are large: each expert opens for
    // about a quarter of the batch, so from B = 512 on a group holds ~128+ rows
    const int* tp256 = B >= kMoePairMinBatch ? ws.tile_prefix256 : nullptr;
    const dim3 sgrid1((Fe + TN - 1) / TN, (B + TM - 1) / TM, G), sgrid2((D + TN - 1) / TN, (B + TM - 1) / TM, G);
    // 3: expert layer 1 over all groups: Hm = Gelu(Sg W1 + b1)
    e = scoped(7 /* RM_K_MOE_GEMM1 */, [&]() -> cudaError_t {
        if (tc)
            return launch_moe_gemm1_tc(ws.Sg, rows_cap, w.W1p, w.b1, ws.Hm, G, D, Fe, ws.counts, ws.offsets,
                                       ws.tile_prefix, tp256, ml.num_sms, ml.err, kMoeWaitTimeoutNs, s);
        if (ml.act == Act::BF16)
            moe_gemm_simt_kernel<__half, 1><<<sgrid1, 256, 0, s>>>((const __half*)ws.Sg, (const __half*)w.W1p, w.b1,
                                                                   (__half*)ws.Hm, ws.counts, ws.offsets, nullptr,
                                                                   Fe, D);
        else
            moe_gemm_simt_kernel<float, 1><<<sgrid1, 256, 0, s>>>((const float*)ws.Sg, (const float*)w.W1p, w.b1,
                                                                  (float*)ws.Hm, ws.counts, ws.offsets, nullptr, Fe,
                                                                  D);
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    // 4: expert layer 2 over all groups: Y = gate (Hm W2 + b2), one packed row per open
    //    (b, t, e), written over the gathered rows (no longer needed)
    e = scoped(8 /* RM_K_MOE_GEMM2 */, [&]() -> cudaError_t {
        if (tc)
            return launch_moe_gemm2_tc(ws.Hm, rows_cap, w.W2p, w.b2, ws.Sg, G, D, Fe, ws.counts, ws.offsets,
                                       ws.tile_prefix, tp256, ws.row_gate, ml.num_sms, ml.err, kMoeWaitTimeoutNs, s);
        if (ml.act == Act::BF16)
            moe_gemm_simt_kernel<__half, 2><<<sgrid2, 256, 0, s>>>((const __half*)ws.Hm, (const __half*)w.W2p, w.b2,
                                                                   (__half*)ws.Sg, ws.counts, ws.offsets, ws.row_gate,
                                                                   D, Fe);
        else
            moe_gemm_simt_kernel<float, 2><<<sgrid2, 256, 0, s>>>((const float*)ws.Hm, (const float*)w.W2p, w.b2,
                                                                  (float*)ws.Sg, ws.counts, ws.offsets, ws.row_gate,
                                                                  D, Fe);
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    // 5: V[b, t] = sum of the open experts' rows, ascending e
    return scoped(10 /* RM_K_MOE_COMBINE */, [&]() -> cudaError_t {
        int grid = (int)(((long long)B * T * 32 + 255) / 256);
        if (grid > ml.num_sms * 16) grid = ml.num_sms * 16;
        const bool vec = D % 8 == 0 && (v_sb % 4 == 0) && (v_st % 4 == 0) && ((uintptr_t)V % 16 == 0);
        if (ml.act == Act::BF16 && vec && D % 256 == 0 && D <= 8 * 256) {
            const __half* Y = (const __half*)ws.Sg;
            switch (D / 256) {
                case 1: combine_rows_kernel<1><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                case 2: combine_rows_kernel<2><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                case 3: combine_rows_kernel<3><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                case 4: combine_rows_kernel<4><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                case 5: combine_rows_kernel<5><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                case 6: combine_rows_kernel<6><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                case 7: combine_rows_kernel<7><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
                default: combine_rows_kernel<8><<<grid, 256, 0, s>>>(Y, ws.slot_of, V, v_sb, v_st, B, T, D, E, ws.Bcap); break;
            }
        } else if (ml.act == Act::BF16) {
            if (vec)
                combine_kernel<__half, 8><<<grid, 256, 0, s>>>((const __half*)ws.Sg, ws.slot_of, V, v_sb, v_st, B, T,
                                                               D, E, ws.Bcap);
            else
                combine_kernel<__half, 1><<<grid, 256, 0, s>>>((const __half*)ws.Sg, ws.slot_of, V, v_sb, v_st, B, T,
                                                               D, E, ws.Bcap);
        } else {
            if (vec)
                combine_kernel<float, 4><<<grid, 256, 0, s>>>((const float*)ws.Sg, ws.slot_of, V, v_sb, v_st, B, T,
                                                              D, E, ws.Bcap);
            else
                combine_kernel<float, 1><<<grid, 256, 0, s>>>((const float*)ws.Sg, ws.slot_of, V, v_sb, v_st, B, T,
                                                              D, E, ws.Bcap);
        }
        return cudaGetLastError();
    });
}

cudaError_t moe_residual_z(Act act, const float* V, const void* S, void* Z, int B, int T, int D, int Bcap,
                           cudaStream_t s) {
    const long long n = (long long)T * B * D;
    constexpr int kGridStrideCap = 152 * 16;   // blocks of the grid-stride loop (it strides; a launch-size bound)
    int grid = (int)((n + 255) / 256);
    if (grid > kGridStrideCap) grid = kGridStrideCap;
    if (act == Act::BF16)
        residual_z_kernel<__half><<<grid, 256, 0, s>>>(V, (const __half*)S, (__half*)Z, B, T, D, Bcap);
    else
        residual_z_kernel<float><<<grid, 256, 0, s>>>(V, (const float*)S, (float*)Z, B, T, D, Bcap);
    return cudaGetLastError();
}


// ---- gates of a second router (the inference router during DTSI training) ----------
// One warp per (b, t) row, experts in groups of 8: lane-strided dot products
// over D, then a butterfly sum per expert; lane 0 writes ReLU(. + bg).
namespace {
template <typename Tin>
__global__ void __launch_bounds__(256)
router_gates_kernel(const Tin* __restrict__ S, const float* __restrict__ Wg, const float* __restrict__ bg,
                    float* __restrict__ G, int B, int T, int D, int E) {
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * T;
    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += (long long)gridDim.x * 8) {
        const int t = (int)(row % T);
        const Tin* s = S + (size_t)row * D;
        for (int e0 = 0; e0 < E; e0 += 8) {
            const int ne = min(8, E - e0);
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
            for (int k = lane; k < D; k += 32) {
                const float x = to_f32(s[k]);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < ne) acc[j] = fmaf(x, __ldg(Wg + ((size_t)t * E + e0 + j) * D + k), acc[j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = warp_sum(acc[j]);
            if (lane == 0)
                for (int j = 0; j < ne; ++j)
                    G[(size_t)row * E + e0 + j] = fmaxf(acc[j] + __ldg(bg + (size_t)t * E + e0 + j), 0.f);
        }
    }
}

__global__ void gate_lreg_kernel(const float* __restrict__ G, float* __restrict__ lreg, int B, int TE) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const float* g = G + (size_t)b * TE;
    float s = 0.f;
    for (int i = 0; i < TE; ++i) s += g[i];
    lreg[b] = s;
}

__global__ void __launch_bounds__(256)
gate_activation_kernel(const float* __restrict__ G, float* __restrict__ A, long long rows, int E) {
    __shared__ float red[256];
    const int e = blockIdx.x;
    float s = 0.f;
    for (long long r = threadIdx.x; r < rows; r += 256) s += G[(size_t)r * E + e];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) A[e] = red[0];
}
}  // namespace

cudaError_t moe_router_gates(Act act, const void* S, const float* Wg, const float* bg, float* G, int B, int T,
                             int D, int E, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    long long g = ((long long)B * T + 7) / 8;
    const int grid = (int)(g > 8192 ? 8192 : g);
    if (act == Act::F32)
        router_gates_kernel<float><<<grid, 256, 0, s>>>((const float*)S, Wg, bg, G, B, T, D, E);
    else
        router_gates_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)S, Wg, bg, G, B, T, D, E);
    return cudaGetLastError();
}

cudaError_t moe_gate_sums(const float* G, float* lreg, float* A, int B, int T, int E, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (lreg) {
        gate_lreg_kernel<<<(B + 255) / 256, 256, 0, s>>>(G, lreg, B, T * E);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (A) {
        gate_activation_kernel<<<E, 256, 0, s>>>(G, A, (long long)B * T, E);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace rm
