// Memory-bound kernels of the RankMixer block: TokenMixing fused with the
// first residual and LayerNorm, the second LayerNorm's finalisation (into the
// next layer's mixing, into a [B][T][D] output, or into mean pooling), and
// the small layout/packing kernels used at context creation.
//
// "RankMixer: Scaling Up Ranking Models in Industrial Recommenders", section
// 3.1 Eq. 1 and section 3.3.1 Eq. 3-5; "RankMixer 详解（1）" section 3.1 (the
// element map of the mixing) and section 3.3 (LayerNorm).
//
// Types: Tin is the caller's activation dtype (bf16 or float), Top the
// operand type of the GEMMs (fp16 for bf16 contexts, float for float32
// contexts).  The pre-LN2 rows Z are stored in Top as well.
#include <cstdlib>
#include <type_traits>

#include "rm_common.cuh"
#include "rm_internal.h"
#include "rm_train.h"
#include "rm_unimix.h"

namespace rm {
namespace {

constexpr int kMaxT = 128;

// LN affine applied to a finalised row element.  Every kernel that finalises
// LN2 (the next layer's mixing, the block output, the pool) uses this exact
// expression, so they all see the same float32 value of X_n.
__device__ __forceinline__ float ln_apply(float z, float mean, float rstd, float g, float b) {
    const float n = (z - mean) * rstd;
    return fmaf(n, g, b);
}

template <typename T> struct Vec2;
template <> struct Vec2<float> {
    using type = float2;
    __device__ static float2 load(const float* p) { return *reinterpret_cast<const float2*>(p); }
    __device__ static void store(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
    __device__ static void split(float2 v, float& a, float& b) { a = v.x; b = v.y; }
};
template <> struct Vec2<__half> {
    using type = __half2;
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
    using type = __nv_bfloat162;
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

template <typename T>
__device__ __forceinline__ void load_pair(const T* p, float& a, float& b) {
    Vec2<T>::split(Vec2<T>::load(p), a, b);
}

// Row statistics of the T rows of sample b into shared memory (one warp per row).
__device__ __forceinline__ void sample_row_stats(const MixLnArgs& a, int b, float* s_mean, float* s_rstd, int warp,
                                                 int nwarps, int lane) {
    for (int t = warp; t < a.T; t += nwarps) {
        float mean, rstd;
        merge_row_stats(a.stats + ((size_t)t * a.Bcap + b) * a.nchunk, a.nchunk, a.cw, a.D, a.eps, lane, mean, rstd);
        if (lane == 0) {
            s_mean[t] = mean;
            s_rstd[t] = rstd;
        }
    }
}

// One output row h of the fused mix + residual + LN1, column pairs per lane:
//   y[j] = X[t][h q + r] + X[h][j],  j = t q + r
// X (T rows of length D at stride xrow) is read through `xs` (shared or global
// memory) in its stored type Tx and, when FROM_Z, finalised from pre-LN2
// values.  y stays in registers; S[h] = LN1(y) is stored at srow in the
// operand type Top.  Needs q even and D % 64 == 0.
template <typename Tx, typename Top, bool FROM_Z, int NI>
__device__ __forceinline__ void mix_row_pairs(const MixLnArgs& a, const Tx* xs, size_t xrow, int h,
                                              const float* s_mean, const float* s_rstd, Top* srow, int lane) {
    const int D = a.D, q = a.q;
    const int ni = D >> 6;
    const Tx* xh = xs + (size_t)h * xrow;
    float y[2 * NI];
    float sum = 0.f;
    int t = (2 * lane) / q;
    int r = 2 * lane - t * q;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        if (i < ni) {
            const int j = (i << 6) + (lane << 1);
            const int c = h * q + r;
            float m0, m1, x0, x1;
            load_pair(xs + (size_t)t * xrow + c, m0, m1);
            load_pair(xh + j, x0, x1);
            if (FROM_Z) {
                const float2 gm = *reinterpret_cast<const float2*>(a.g2 + c);
                const float2 bm = *reinterpret_cast<const float2*>(a.be2 + c);
                const float2 gx = *reinterpret_cast<const float2*>(a.g2 + j);
                const float2 bx = *reinterpret_cast<const float2*>(a.be2 + j);
                const float mt = s_mean[t], rt = s_rstd[t], mh = s_mean[h], rh = s_rstd[h];
                m0 = ln_apply(m0, mt, rt, gm.x, bm.x);
                m1 = ln_apply(m1, mt, rt, gm.y, bm.y);
                x0 = ln_apply(x0, mh, rh, gx.x, bx.x);
                x1 = ln_apply(x1, mh, rh, gx.y, bx.y);
            }
            y[2 * i] = m0 + x0;
            y[2 * i + 1] = m1 + x1;
            sum += y[2 * i] + y[2 * i + 1];
            r += 64;                      // next j is 64 columns further
            while (r >= q) {
                r -= q;
                ++t;
            }
        }
    }
    const float mean = warp_sum(sum) / (float)D;
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
        if (i < ni) {
            const float d0 = y[2 * i] - mean, d1 = y[2 * i + 1] - mean;
            sq += d0 * d0 + d1 * d1;
        }
    const float rstd = rsqrtf(warp_sum(sq) / (float)D + a.eps);
#pragma unroll
    for (int i = 0; i < NI; ++i)
        if (i < ni) {
            const int j = (i << 6) + (lane << 1);
            const float2 g = *reinterpret_cast<const float2*>(a.g1 + j);
            const float2 be = *reinterpret_cast<const float2*>(a.be1 + j);
            Vec2<Top>::store(srow + j, ln_apply(y[2 * i], mean, rstd, g.x, be.x),
                             ln_apply(y[2 * i + 1], mean, rstd, g.y, be.y));
        }
}

// ---------------------------------------------------------------------------
// Staged mix + LN1 (bf16 contexts, q even, D % 64 == 0).  Persistent CTAs
// walk samples b = blockIdx.x, + gridDim.x, ...; each sample's T x D source
// rows (the caller's bf16 X, or the previous layer's fp16 pre-LN2 rows Z) are
// brought into shared memory with 1-D bulk copies on an mbarrier, double
// buffered so the next sample's copy overlaps this sample's arithmetic.
// ---------------------------------------------------------------------------
template <typename Tsrc, bool FROM_Z, int NI>
__global__ void __launch_bounds__(512)
mix_ln1_staged_kernel(const MixLnArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int T = a.T, D = a.D;
    const uint32_t row_bytes = (uint32_t)D * 2u;
    const uint32_t buf_bytes = (uint32_t)T * row_bytes;
    Tsrc* buf = reinterpret_cast<Tsrc*>(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * (size_t)buf_bytes);
    float* s_mean = reinterpret_cast<float*>(bars + 2);
    float* s_rstd = s_mean + kMaxT;
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_rstd + kMaxT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const Tsrc* src = FROM_Z ? reinterpret_cast<const Tsrc*>(a.Z) : reinterpret_cast<const Tsrc*>(a.X);
    __half* S = reinterpret_cast<__half*>(a.S);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_next();

    auto issue = [&](int b, int slot) {   // thread 0 only
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(buf) + (uint32_t)slot * buf_bytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, buf_bytes);
        if (!FROM_Z) {
            bulk_copy_g2s(dst, src + (size_t)b * T * D, buf_bytes, bar);
        } else {
            for (int t = 0; t < T; ++t)
                bulk_copy_g2s(dst + (uint32_t)t * row_bytes, src + ((size_t)t * a.Bcap + b) * D, row_bytes, bar);
        }
    };

    if (threadIdx.x == 0 && (int)blockIdx.x < a.B) issue(blockIdx.x, 0);
    int it = 0;
    for (int b = blockIdx.x; b < a.B; b += gridDim.x, ++it) {
        const int slot = it & 1;
        if (threadIdx.x == 0 && b + (int)gridDim.x < a.B) issue(b + gridDim.x, slot ^ 1);
        if (FROM_Z) sample_row_stats(a, b, s_mean, s_rstd, warp, nwarps, lane);
        mbar_wait_bounded(smem_u32(&bars[slot]), (uint32_t)(it >> 1) & 1u, s_abort, a.err, a.timeout_ns);
        __syncthreads();
        if (*s_abort) break;
        const Tsrc* xs = buf + (size_t)slot * T * D;
        for (int h = warp; h < T; h += nwarps)
            mix_row_pairs<Tsrc, __half, FROM_Z, NI>(a, xs, (size_t)D, h, s_mean, s_rstd,
                                                     S + ((size_t)h * a.Bcap + b) * D, lane);
        __syncthreads();    // the slot and the row statistics are reused by later samples
    }
}

// ---------------------------------------------------------------------------
// Staged mix + LN1, 8 columns per lane (bf16 contexts, q % 8 == 0,
// D % 256 == 0).  Same pipeline as above, with:
//   - 16-byte shared-memory loads and global stores (8 elements per lane);
//     an 8-column group never crosses a head block because q % 8 == 0;
//   - both LN affines staged in shared memory once per CTA;
//   - (FROM_Z) LN2 finalised in place, once per element, before mixing.
// ---------------------------------------------------------------------------
// Shared-memory layout of the 8-wide kernel.  Each staged row of D 16-bit
// elements is padded to a stride RS with RS = q (mod 64): an 8-lane phase of a
// 16-byte load covers 64 consecutive mixed columns, which may span two source
// rows (head h of row t, then head h of row t + 1); with this stride the second
// row's chunks continue the first row's bank sequence, so the phase touches 8
// distinct 16-byte bank groups.  The LN affines are kept as fp16 (exact: they
// arrive as bf16 values), so a lane's 8 affines are one 16-byte load.
__host__ __device__ __forceinline__ int v8_row_stride(int D, int q) { return D + (q & 63); }

// A 32-bit word of two 16-bit values (bf16 or fp16, low half first) -> packed fp32 pair.
template <bool BF16>
__device__ __forceinline__ uint64_t pair16_to_f2(uint32_t w) {
    if constexpr (BF16) {
        return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        return f2_pack(f.x, f.y);
    }
}

// Two row buffers, the four fp16 affines, two mbarriers, the row mean / rstd
// arrays and the abort flag.
size_t v8_smem_bytes(int T, int D, int q) {
    return 2 * (size_t)T * v8_row_stride(D, q) * 2 + 4 * (size_t)D * 2 + 16 + 2 * kMaxT * 4 + 16;
}

// DBG (test hook): write the residual sum y = Mix(X) + X as float32 to
// a.Ydbg instead of LN1; with FROM_Z the LN2 finalisation runs with mean 0,
// rstd 1, gamma 1, beta 0 (the identity on fp16 values), so the gather and
// the fp16 sum are checked bit for bit.
template <bool FROM_Z, int NV, bool DBG = false>
__global__ void __launch_bounds__(512)
mix_ln1_v8_kernel(const MixLnArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int T = a.T, D = a.D, q = a.q;
    const int RS = v8_row_stride(D, q);
    const uint32_t row_bytes = (uint32_t)D * 2u;
    const uint32_t buf_elems = (uint32_t)T * RS;
    uint16_t* buf = reinterpret_cast<uint16_t*>(smem);                       // [2][T][RS] 16-bit
    __half* sg1 = reinterpret_cast<__half*>(smem + 4 * (size_t)buf_elems);    // [D] each
    __half* sb1 = sg1 + D;
    __half* sg2 = sb1 + D;                                                    // FROM_Z only
    __half* sb2 = sg2 + D;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb2 + D);
    float* s_mean = reinterpret_cast<float*>(bars + 2);
    float* s_rstd = s_mean + kMaxT;
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_rstd + kMaxT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const uint16_t* src = FROM_Z ? reinterpret_cast<const uint16_t*>(a.Z) : reinterpret_cast<const uint16_t*>(a.X);
    __half* S = reinterpret_cast<__half*>(a.S);

    for (int j = threadIdx.x; j < D; j += blockDim.x) {
        if constexpr (DBG) {
            sg2[j] = __float2half_rn(1.0f);
            sb2[j] = __float2half_rn(0.0f);
            continue;
        }
        sg1[j] = __float2half_rn(a.g1[j]);
        sb1[j] = __float2half_rn(a.be1[j]);
        if (FROM_Z) {
            sg2[j] = __float2half_rn(a.g2[j]);
            sb2[j] = __float2half_rn(a.be2[j]);
        }
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();              // the layer input and its statistics come from the previous kernel
    pdl_launch_next();

    auto issue = [&](int b, int slot) {   // warp 0: lane 0 arms the barrier, lane t copies row t
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(buf) + (uint32_t)slot * buf_elems * 2u;
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)T * row_bytes);
        __syncwarp();
        for (int t = lane; t < T; t += 32) {
            const uint16_t* row = FROM_Z ? src + ((size_t)t * a.Bcap + b) * D : src + ((size_t)b * T + t) * D;
            // (a skipped copy leaves the barrier short: the bounded wait then ends the sample)
            if (RM_IN_BOUNDS(b >= 0 && b < a.B && b < a.Bcap, a.err))
                bulk_copy_g2s(dst + (uint32_t)t * (uint32_t)RS * 2u, row, row_bytes, bar);
        }
    };

    // FROM_Z with merged row statistics (one (mean, M2) per row): lane k of warp w
    // holds row w + k nwarps of the next sample, loaded one sample ahead
    const bool merged = FROM_Z && (DBG || a.nchunk == 1);
    const int pre_t = warp + lane * nwarps;
    const bool pre_lane = merged && pre_t < T;
    float2 pre = make_float2(0.f, 0.f);
    // work items w = (sample w / rsplit, output rows of part w % rsplit); with small
    // batches a sample's rows are spread over rsplit CTAs (each stages the whole sample)
    const int rsplit = a.rsplit > 0 ? a.rsplit : 1;
    const int nitems = a.B * rsplit;
    if (!DBG && pre_lane && (int)blockIdx.x < nitems)
        pre = __ldg(a.stats + (size_t)pre_t * a.Bcap + (int)blockIdx.x / rsplit);

    // the lane's gather offsets inside a staged sample, one per 8-column group i:
    // output column j0 = 256 i + 8 lane of row h reads row t = j0 / q at column
    // h q + (j0 - t q) -- the same t and remainder for every row h and sample
    int goff[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j0 = (i << 8) + (lane << 3);
        const int t = j0 / q;
        goff[i] = t * RS + (j0 - t * q);
    }

    if (warp == 0 && (int)blockIdx.x < nitems) issue((int)blockIdx.x / rsplit, 0);
    int it = 0;
    for (int w = blockIdx.x; w < nitems; w += gridDim.x, ++it) {
        const int b = w / rsplit, part = w - b * rsplit;
        const int bn = (w + (int)gridDim.x) / rsplit;          // sample of this CTA's next item
        const int slot = it & 1;
        if (warp == 0 && w + (int)gridDim.x < nitems) issue(bn, slot ^ 1);
        if (merged) {
            if (pre_lane && DBG) {
                s_mean[pre_t] = 0.0f;
                s_rstd[pre_t] = 1.0f;
            } else if (pre_lane) {
                s_mean[pre_t] = pre.x;
                s_rstd[pre_t] = rsqrtf(pre.y / (float)D + a.eps);
                if (w + (int)gridDim.x < nitems) pre = __ldg(a.stats + (size_t)pre_t * a.Bcap + bn);
            }
        } else if (FROM_Z) {
            sample_row_stats(a, b, s_mean, s_rstd, warp, nwarps, lane);
        }
        mbar_wait_bounded(smem_u32(&bars[slot]), (uint32_t)(it >> 1) & 1u, s_abort, a.err, a.timeout_ns);
        __syncthreads();
        if (*s_abort) break;
        uint16_t* xs = buf + (size_t)slot * buf_elems;
        if (FROM_Z) {
            // X_{n-1} = LN2(Z) in place (fp16), 8 columns per thread: a thread keeps one
            // 8-column group (its gamma2 / beta2 loaded once) and walks every nsl-th
            // row, so the affines cost one shared-memory load per group instead of
            // one per group and row; rows are loaded four at a time before use.
            // (z - mean) (rstd gamma) + beta on fp16 pairs: the result is stored in
            // fp16, and the row statistics themselves were merged in fp32.
            const int ngr = D >> 3;
            const int nsl = blockDim.x >= ngr ? (int)blockDim.x / ngr : 1;
            for (int wi = threadIdx.x; wi < ngr * nsl; wi += blockDim.x) {
                const int cg = wi % ngr, sl = wi / ngr;
                const int c = cg << 3;
                const uint4 gv = *reinterpret_cast<const uint4*>(sg2 + c);
                const uint4 bv = *reinterpret_cast<const uint4*>(sb2 + c);
                const __half2* g2h = reinterpret_cast<const __half2*>(&gv);
                const __half2* b2h = reinterpret_cast<const __half2*>(&bv);
                for (int t0 = sl; t0 < T; t0 += 4 * nsl) {
                    uint4 zv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = t0 + u * nsl;
                        if (t < T) zv[u] = *reinterpret_cast<const uint4*>(xs + (size_t)t * RS + c);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = t0 + u * nsl;
                        if (t < T) {
                            const __half2 m2 = __float2half2_rn(s_mean[t]), r2 = __float2half2_rn(s_rstd[t]);
                            __half2* z2 = reinterpret_cast<__half2*>(&zv[u]);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                z2[k] = __hfma2(__hsub2(z2[k], m2), __hmul2(r2, g2h[k]), b2h[k]);
                            *reinterpret_cast<uint4*>(xs + (size_t)t * RS + c) = zv[u];
                        }
                    }
                }
            }
            __syncthreads();
        }
        // mix + residual + LN1 on packed fp32 pairs: y = m + x and the row
        // statistics in float32; the affine (y - mean) rstd gamma + beta as one
        // float32 pair fma to (y - mean) rstd, then one fp16 pair fma with the fp16
        // gamma, beta (S is stored in fp16)
        const int nv = D >> 8;
        const int h0 = part * T / rsplit, h1 = (part + 1) * T / rsplit;
        for (int h = h0 + warp; h < h1; h += nwarps) {
            const uint16_t* xh = xs + (size_t)h * RS;
            uint64_t y[4 * NV];
            uint64_t s2 = f2_splat(0.f);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (i < nv) {
                    const int j0 = (i << 8) + (lane << 3);
                    const bool gok = RM_IN_BOUNDS(goff[i] + h * q + 8 <= T * RS && j0 + 8 <= RS, a.err);
                    const uint4 mv = gok ? *reinterpret_cast<const uint4*>(xs + goff[i] + h * q)
                                         : make_uint4(0u, 0u, 0u, 0u);
                    const uint4 xv = gok ? *reinterpret_cast<const uint4*>(xh + j0) : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if constexpr (FROM_Z) {     // fp16 rows: add in fp16, convert once
                            const __half2 yh = __hadd2(*reinterpret_cast<const __half2*>(&mw[k]),
                                                       *reinterpret_cast<const __half2*>(&xw[k]));
                            const float2 yf = __half22float2(yh);
                            y[4 * i + k] = f2_pack(yf.x, yf.y);
                        } else {
                            y[4 * i + k] = f2_add(pair16_to_f2<true>(mw[k]), pair16_to_f2<true>(xw[k]));
                        }
                        s2 = f2_add(s2, y[4 * i + k]);
                    }
                }
            }
            if constexpr (DBG) {
                float* yrow = a.Ydbg + ((size_t)h * a.Bcap + b) * D;
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    if (i < nv) {
                        const int j0 = (i << 8) + (lane << 3);
                        float o[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) f2_unpack(y[4 * i + k], o[2 * k], o[2 * k + 1]);
                        if (RM_IN_BOUNDS(b < a.Bcap && j0 + 8 <= D, a.err)) {
                            reinterpret_cast<float4*>(yrow + j0)[0] = make_float4(o[0], o[1], o[2], o[3]);
                            reinterpret_cast<float4*>(yrow + j0)[1] = make_float4(o[4], o[5], o[6], o[7]);
                        }
                    }
                continue;
            }
            float lo, hi;
            f2_unpack(s2, lo, hi);
            const float mean = warp_sum(lo + hi) / (float)D;
            const uint64_t nmean2 = f2_splat(-mean);
            uint64_t q2 = f2_splat(0.f);
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (i < nv) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t d = f2_add(y[4 * i + k], nmean2);
                        q2 = f2_fma(d, d, q2);
                    }
                }
            f2_unpack(q2, lo, hi);
            const float rstd = rsqrtf(warp_sum(lo + hi) / (float)D + a.eps);
            const uint64_t rstd2 = f2_splat(rstd), nmr2 = f2_splat(-mean * rstd);
            __half* srow = S + ((size_t)h * a.Bcap + b) * D;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (i < nv) {
                    const int j0 = (i << 8) + (lane << 3);
                    const uint4 gv = *reinterpret_cast<const uint4*>(sg1 + j0);
                    const uint4 bv = *reinterpret_cast<const uint4*>(sb1 + j0);
                    const __half2* g2h = reinterpret_cast<const __half2*>(&gv);
                    const __half2* b2h = reinterpret_cast<const __half2*>(&bv);
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t nh = pack_f16x2_from_f2(f2_fma(y[4 * i + k], rstd2, nmr2));
                        const __half2 v = __hfma2(*reinterpret_cast<const __half2*>(&nh), g2h[k], b2h[k]);
                        o[k] = *reinterpret_cast<const uint32_t*>(&v);
                    }
                    if (RM_IN_BOUNDS(b < a.Bcap && j0 + 8 <= D, a.err))
                        *reinterpret_cast<uint4*>(srow + j0) = make_uint4(o[0], o[1], o[2], o[3]);
                }
        }
        __syncthreads();    // the slot and the row statistics are reused by later samples
    }
}

bool v8_ok(bool, const MixLnArgs& a) {
    return a.q % 8 == 0 && a.D % 256 == 0 && a.D <= 3072 && a.T <= kMaxT && v8_smem_bytes(a.T, a.D, a.q) <= 226 * 1024;
}

template <bool FROM_Z, int NV, bool DBG = false>
cudaError_t launch_v8(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    auto k = mix_ln1_v8_kernel<FROM_Z, NV, DBG>;
    const size_t smem = v8_smem_bytes(a.T, a.D, a.q);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int threads = 32 * (a.T < 16 ? a.T : 16);
    if (threads < 128) threads = 128;
    int per_sm = 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    // small batches: spread each sample's output rows over several CTAs (at least
    // two rows each) so that more SMs work on it
    MixLnArgs b = a;
    const int slots = num_sms * per_sm;
    b.rsplit = 1;
    if (a.B < slots) {
        int r = slots / a.B;
        if (r > a.T / 2) r = a.T / 2;
        b.rsplit = r > 1 ? r : 1;
    }
    int grid = slots;
    if (grid > a.B * b.rsplit) grid = a.B * b.rsplit;
    return launch_k(k, dim3(grid), dim3(threads), smem, s, b);
}

template <bool FROM_Z, bool DBG = false>
cudaError_t launch_v8_dispatch(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    const int nv = a.D / 256;
    if (nv <= 1) return launch_v8<FROM_Z, 1, DBG>(a, num_sms, s);
    if (nv <= 2) return launch_v8<FROM_Z, 2, DBG>(a, num_sms, s);
    if (nv <= 3) return launch_v8<FROM_Z, 3, DBG>(a, num_sms, s);
    if (nv <= 4) return launch_v8<FROM_Z, 4, DBG>(a, num_sms, s);
    if (nv <= 6) return launch_v8<FROM_Z, 6, DBG>(a, num_sms, s);
    if (nv <= 8) return launch_v8<FROM_Z, 8, DBG>(a, num_sms, s);
    return launch_v8<FROM_Z, 12, DBG>(a, num_sms, s);
}

// ---------------------------------------------------------------------------
// Direct mix + LN1 (float32 contexts and shapes the staged kernel does not
// take): X read straight from global memory, one CTA per sample.
// VEC = 2 uses mix_row_pairs (q even, D % 64 == 0); VEC = 1 handles any q.
// ---------------------------------------------------------------------------
constexpr int kMixThreads = 256;
constexpr int kMixWarps = kMixThreads / 32;

template <typename Tin, typename Top, bool FROM_Z, int VEC, int NI>
__global__ void __launch_bounds__(kMixThreads)
mix_ln1_direct_kernel(const MixLnArgs a) {
    __shared__ float s_mean[kMaxT], s_rstd[kMaxT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, D = a.D, q = a.q;
    Top* S = reinterpret_cast<Top*>(a.S);
    pdl_wait();
    pdl_launch_next();
    for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        // source rows: X sample-major (row stride D) or Z token-major (row stride Bcap D)
        const Tin* X = reinterpret_cast<const Tin*>(a.X) + (size_t)b * T * D;
        const Top* Z = reinterpret_cast<const Top*>(a.Z) + (size_t)b * D;
        const size_t zrow = (size_t)a.Bcap * D;
        if (FROM_Z) {
            sample_row_stats(a, b, s_mean, s_rstd, warp, kMixWarps, lane);
            __syncthreads();
        }
        for (int h = warp; h < T; h += kMixWarps) {
            Top* srow = S + ((size_t)h * a.Bcap + b) * D;
            if (VEC == 2) {
                if (FROM_Z)
                    mix_row_pairs<Top, Top, true, NI>(a, Z, zrow, h, s_mean, s_rstd, srow, lane);
                else
                    mix_row_pairs<Tin, Top, false, NI>(a, X, (size_t)D, h, s_mean, s_rstd, srow, lane);
                continue;
            }
            auto load1 = [&](int t, int c) -> float {
                if (FROM_Z) return ln_apply(to_f32(Z[t * zrow + c]), s_mean[t], s_rstd[t], a.g2[c], a.be2[c]);
                return to_f32(X[(size_t)t * D + c]);
            };
            float y[NI];
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int j = (i << 5) + lane;
                if (j < D) {
                    const int t = j / q;
                    const int r = j - t * q;
                    y[i] = load1(t, h * q + r) + load1(h, j);
                    sum += y[i];
                }
            }
            const float mean = warp_sum(sum) / (float)D;
            float sq = 0.f;
#pragma unroll
            for (int i = 0; i < NI; ++i)
                if ((i << 5) + lane < D) {
                    const float d = y[i] - mean;
                    sq += d * d;
                }
            const float rstd = rsqrtf(warp_sum(sq) / (float)D + a.eps);
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int j = (i << 5) + lane;
                if (j < D) srow[j] = from_f32<Top>(ln_apply(y[i], mean, rstd, a.g1[j], a.be1[j]));
            }
        }
        if (FROM_Z) __syncthreads();   // s_mean / s_rstd are rewritten for the next sample
    }
}

template <typename Tin, typename Top, bool FROM_Z, int VEC, int NI>
cudaError_t launch_direct(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    int grid = num_sms * 8;
    if (grid > a.B) grid = a.B;
    return launch_k(mix_ln1_direct_kernel<Tin, Top, FROM_Z, VEC, NI>, dim3(grid), dim3(kMixThreads), 0, s, a);
}

template <typename Tin, typename Top, bool FROM_Z>
cudaError_t launch_direct_dispatch(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    const bool vec2 = (a.q % 2 == 0) && (a.D % 64 == 0);
    if (vec2) {
        const int ni = a.D / 64;
        if (ni <= 4) return launch_direct<Tin, Top, FROM_Z, 2, 4>(a, num_sms, s);
        if (ni <= 12) return launch_direct<Tin, Top, FROM_Z, 2, 12>(a, num_sms, s);
        if (ni <= 24) return launch_direct<Tin, Top, FROM_Z, 2, 24>(a, num_sms, s);
        if (ni <= 48) return launch_direct<Tin, Top, FROM_Z, 2, 48>(a, num_sms, s);
        return cudaErrorNotSupported;
    }
    const int ni = (a.D + 31) / 32;
    if (ni <= 8) return launch_direct<Tin, Top, FROM_Z, 1, 8>(a, num_sms, s);
    if (ni <= 48) return launch_direct<Tin, Top, FROM_Z, 1, 48>(a, num_sms, s);
    return cudaErrorNotSupported;
}

size_t staged_smem_bytes(int T, int D) { return 2 * (size_t)T * D * 2 + 16 + 2 * kMaxT * 4 + 16; }

template <typename Tsrc, bool FROM_Z, int NI>
cudaError_t launch_staged(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    auto k = mix_ln1_staged_kernel<Tsrc, FROM_Z, NI>;
    const size_t smem = staged_smem_bytes(a.T, a.D);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int threads = 32 * (a.T < 16 ? a.T : 16);
    if (threads < 128) threads = 128;
    int per_sm = 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int grid = num_sms * per_sm;
    if (grid > a.B) grid = a.B;
    return launch_k(k, dim3(grid), dim3(threads), smem, s, a);
}

template <typename Tsrc, bool FROM_Z>
cudaError_t launch_staged_dispatch(const MixLnArgs& a, int num_sms, cudaStream_t s) {
    const int ni = a.D / 64;
    if (ni <= 4) return launch_staged<Tsrc, FROM_Z, 4>(a, num_sms, s);
    if (ni <= 12) return launch_staged<Tsrc, FROM_Z, 12>(a, num_sms, s);
    if (ni <= 24) return launch_staged<Tsrc, FROM_Z, 24>(a, num_sms, s);
    return launch_staged<Tsrc, FROM_Z, 48>(a, num_sms, s);
}

bool staged_ok(const MixLnArgs& a) {
    return a.q % 2 == 0 && a.D % 64 == 0 && a.D <= 3072 && a.T <= kMaxT &&
           staged_smem_bytes(a.T, a.D) <= 220 * 1024;
}

// ---------------------------------------------------------------------------
// LN2 finalisation into a sample-major output: one warp per (b, t) row.
// ---------------------------------------------------------------------------
template <typename Tz, typename Tout>
__global__ void ln2_out_kernel(const Tz* __restrict__ Z, const float2* __restrict__ stats,
                               const float* __restrict__ g2, const float* __restrict__ be2, Tout* __restrict__ X,
                               int B, int T, int D, int Bcap, int nchunk, int cw, float eps) {
    pdl_wait();
    pdl_launch_next();
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = wid; r < (long long)B * T; r += nw) {
        const int b = (int)(r / T), t = (int)(r % T);
        const size_t zr = (size_t)t * Bcap + b;
        float mean, rstd;
        merge_row_stats(stats + zr * nchunk, nchunk, cw, D, eps, lane, mean, rstd);
        const Tz* z = Z + zr * D;
        Tout* x = X + ((size_t)b * T + t) * D;
        for (int j = lane; j < D; j += 32)
            x[j] = from_f32<Tout>(ln_apply(to_f32(z[j]), mean, rstd, g2[j], be2[j]));
    }
}

// The same for fp16 Z and D a multiple of 256: lane l finalises values
// 256 k + 8 l .. + 7 of the row with 16-byte loads and stores (the scalar
// kernel moves 2 bytes per lane per instruction).  Same expression, same
// row statistics: bit-identical outputs.
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&o)[8]) {
    uint4 w;
    w.x = pack_bf16x2(o[0], o[1]);
    w.y = pack_bf16x2(o[2], o[3]);
    w.z = pack_bf16x2(o[4], o[5]);
    w.w = pack_bf16x2(o[6], o[7]);
    *reinterpret_cast<uint4*>(p) = w;
}
__device__ __forceinline__ void store8(__half* p, const float (&o)[8]) {
    uint4 w;
    w.x = pack_f16x2(o[0], o[1]);
    w.y = pack_f16x2(o[2], o[3]);
    w.z = pack_f16x2(o[4], o[5]);
    w.w = pack_f16x2(o[6], o[7]);
    *reinterpret_cast<uint4*>(p) = w;
}
__device__ __forceinline__ void store8(float* p, const float (&o)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(o[4], o[5], o[6], o[7]);
}

template <typename Tout>
__global__ void ln2_out_vec_kernel(const __half* __restrict__ Z, const float2* __restrict__ stats,
                                   const float* __restrict__ g2, const float* __restrict__ be2, Tout* __restrict__ X,
                                   int B, int T, int D, int Bcap, int nchunk, int cw, float eps) {
    pdl_wait();
    pdl_launch_next();
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = wid; r < (long long)B * T; r += nw) {
        const int b = (int)(r / T), t = (int)(r % T);
        const size_t zr = (size_t)t * Bcap + b;
        float mean, rstd;
        merge_row_stats(stats + zr * nchunk, nchunk, cw, D, eps, lane, mean, rstd);
        const __half* z = Z + zr * D;
        Tout* x = X + ((size_t)b * T + t) * D;
        for (int d = 8 * lane; d < D; d += 256) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(z + d));
            const __half2* h = reinterpret_cast<const __half2*>(&v);
            const float4 ga = __ldg(reinterpret_cast<const float4*>(g2 + d));
            const float4 gb = __ldg(reinterpret_cast<const float4*>(g2 + d + 4));
            const float4 ba = __ldg(reinterpret_cast<const float4*>(be2 + d));
            const float4 bb = __ldg(reinterpret_cast<const float4*>(be2 + d + 4));
            const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
            const float be[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
            float o[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __half22float2(h[u]);
                o[2 * u] = ln_apply(f.x, mean, rstd, gg[2 * u], be[2 * u]);
                o[2 * u + 1] = ln_apply(f.y, mean, rstd, gg[2 * u + 1], be[2 * u + 1]);
            }
            store8(x + d, o);
        }
    }
}

// ---------------------------------------------------------------------------
// Last LN2 finalisation + mean pooling over tokens, one CTA per sample.  The
// mean is taken over the float32 LN2 outputs in token order; XL (optional)
// receives them rounded to the caller's dtype.
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 256;
constexpr int kPoolBatch = 8;

template <typename Tz, typename Tout>
__global__ void __launch_bounds__(kPoolThreads, 4)
pool_kernel(const Tz* __restrict__ Z, const float2* __restrict__ stats, const float* __restrict__ g2,
            const float* __restrict__ be2, float* __restrict__ pooled, Tout* __restrict__ XL, int B, int T, int D,
            int Bcap, int nchunk, int cw, float eps) {
    __shared__ float s_mean[kMaxT], s_rstd[kMaxT];
    __shared__ __half2 s_rh[kMaxT], s_nmrh[kMaxT];     // rstd and -mean rstd as fp16 pairs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch_next();
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        for (int t = warp; t < T; t += kPoolThreads / 32) {
            float mean, rstd;
            merge_row_stats(stats + ((size_t)t * Bcap + b) * nchunk, nchunk, cw, D, eps, lane, mean, rstd);
            if (lane == 0) {
                s_mean[t] = mean;
                s_rstd[t] = rstd;
                s_rh[t] = __float2half2_rn(rstd);
                s_nmrh[t] = __float2half2_rn(-mean * rstd);
            }
        }
        __syncthreads();
        if constexpr (std::is_same_v<Tz, __half>) {
            if (XL == nullptr && (D & 1) == 0) {
                // pooled = gamma mean_t((z - mean_t) rstd_t) + beta: the centred, scaled values
                // on fp16 pairs (one fma), summed over kPoolBatch tokens in fp16, each partial
                // sum converted once and added in float32 (token order kept)
                const size_t tstride = (size_t)Bcap * D;
                for (int j = 2 * threadIdx.x; j < D; j += 2 * kPoolThreads) {
                    const __half* zc = Z + (size_t)b * D + j;
                    float acc0 = 0.f, acc1 = 0.f;
                    for (int t0 = 0; t0 < T; t0 += kPoolBatch) {
                        __half2 zz[kPoolBatch];
#pragma unroll
                        for (int u = 0; u < kPoolBatch; ++u)
                            if (t0 + u < T) zz[u] = *reinterpret_cast<const __half2*>(zc + (size_t)(t0 + u) * tstride);
                        __half2 part = __float2half2_rn(0.f);
#pragma unroll
                        for (int u = 0; u < kPoolBatch; ++u)
                            if (t0 + u < T) part = __hadd2(part, __hfma2(zz[u], s_rh[t0 + u], s_nmrh[t0 + u]));
                        const float2 pf = __half22float2(part);
                        acc0 += pf.x;
                        acc1 += pf.y;
                    }
                    const float2 g = *reinterpret_cast<const float2*>(g2 + j);
                    const float2 be = *reinterpret_cast<const float2*>(be2 + j);
                    *reinterpret_cast<float2*>(pooled + (size_t)b * D + j) =
                        make_float2(fmaf(g.x, acc0 / (float)T, be.x), fmaf(g.y, acc1 / (float)T, be.y));
                }
                __syncthreads();
                continue;
            }
        }
        if ((D & 1) == 0) {
            const size_t tstride = (size_t)Bcap * D;
            for (int j = 2 * threadIdx.x; j < D; j += 2 * kPoolThreads) {
                const float2 g = *reinterpret_cast<const float2*>(g2 + j);
                const float2 be = *reinterpret_cast<const float2*>(be2 + j);
                float acc0 = 0.f, acc1 = 0.f;
                const Tz* zc = Z + (size_t)b * D + j;
                // tokens in batches of kPoolBatch: the loads of a batch are issued before its
                // arithmetic, so that several are in flight (the sum keeps token order)
                for (int t0 = 0; t0 < T; t0 += kPoolBatch) {
                    typename Vec2<Tz>::type zz[kPoolBatch];
#pragma unroll
                    for (int u = 0; u < kPoolBatch; ++u)
                        if (t0 + u < T) zz[u] = Vec2<Tz>::load(zc + (size_t)(t0 + u) * tstride);
#pragma unroll
                    for (int u = 0; u < kPoolBatch; ++u) {
                        if (t0 + u < T) {
                            const int t = t0 + u;
                            float z0, z1;
                            Vec2<Tz>::split(zz[u], z0, z1);
                            const float v0 = ln_apply(z0, s_mean[t], s_rstd[t], g.x, be.x);
                            const float v1 = ln_apply(z1, s_mean[t], s_rstd[t], g.y, be.y);
                            if (XL) Vec2<Tout>::store(XL + ((size_t)b * T + t) * D + j, v0, v1);
                            acc0 += v0;
                            acc1 += v1;
                        }
                    }
                }
                *reinterpret_cast<float2*>(pooled + (size_t)b * D + j) = make_float2(acc0 / (float)T, acc1 / (float)T);
            }
        } else {
            for (int j = threadIdx.x; j < D; j += kPoolThreads) {
                const float g = g2[j], be = be2[j];
                float acc = 0.f;
                for (int t = 0; t < T; ++t) {
                    const float v = ln_apply(to_f32(Z[((size_t)t * Bcap + b) * D + j]), s_mean[t], s_rstd[t], g, be);
                    if (XL) XL[((size_t)b * T + t) * D + j] = from_f32<Tout>(v);
                    acc += v;
                }
                pooled[(size_t)b * D + j] = acc / (float)T;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// (mean, M2) of each full row from its nchunk chunk partials (mean, M2 over cw
// columns each), merged by Chan's formula (merge_chunks, the same bits as a
// consumer that merges the partials itself); one thread per row (the rows of
// the first B samples of every token).  Consumers then read one value per row.
// ---------------------------------------------------------------------------
__global__ void stats_finalize_kernel(const float2* __restrict__ part, float2* __restrict__ out, int B, int T,
                                      int Bcap, int nchunk, int cw) {
    pdl_wait();
    pdl_launch_next();
    const long long n = (long long)T * B;
    for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < n; r += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(r / B), b = (int)(r % B);
        out[(size_t)t * Bcap + b] = merge_chunks(part + ((size_t)t * Bcap + b) * nchunk, nchunk, cw);
    }
}

// ---------------------------------------------------------------------------
// Row statistics (mean, M2) of full Z rows, two passes, one warp per row.
// ---------------------------------------------------------------------------
template <typename Tz>
__global__ void rowstats_kernel(const Tz* __restrict__ Z, float2* __restrict__ stats, int B, int T, int D, int Bcap) {
    pdl_wait();
    pdl_launch_next();
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = wid; r < (long long)B * T; r += nw) {
        const int t = (int)(r / B), b = (int)(r % B);
        const size_t zr = (size_t)t * Bcap + b;
        const Tz* z = Z + zr * D;
        float s = 0.f;
        for (int j = lane; j < D; j += 32) s += to_f32(z[j]);
        const float mean = warp_sum(s) / (float)D;
        float m2 = 0.f;
        for (int j = lane; j < D; j += 32) {
            const float d = to_f32(z[j]) - mean;
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

__global__ void debug_gelu_kernel(const float* __restrict__ u, float* __restrict__ out, long long n, int form) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        if (form == 0) {
            out[i] = gelu_erf(u[i]);
        } else {     // the packed form, value in the low half, its neighbour in the high half
            const float nb = i + 1 < n ? u[i + 1] : 0.f;
            float lo, hi;
            f2_unpack(gelu_erf_x2(f2_pack(u[i], nb), f2_pack(0.f, 0.f)), lo, hi);
            out[i] = lo;
        }
    }
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

// Default cap on the blocks of a grid-stride loop (16 per SM of the 152-SM
// part; the loops stride, so the cap only bounds the launch size).
constexpr int kGridStrideCap = 152 * 16;

inline int grid_for(long long n, int threads, int cap = kGridStrideCap) {
    long long g = (n + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

// Pooled output only (no X_L), fp16 Z, D % 8 == 0: the same fp16-pair sums as
// pool_kernel's first branch with 16-byte loads, thread l owning columns
// 8 l .. 8 l + 7 and a CTA of D / 8 threads per sample, so that several
// CTAs per SM keep more loads in flight.  Same operations in the same order:
// bit-identical to pool_kernel.
template <int TB>
__global__ void __launch_bounds__(256)
pool_vec_kernel(const __half* __restrict__ Z, const float2* __restrict__ stats, const float* __restrict__ g2,
                const float* __restrict__ be2, float* __restrict__ pooled, int B, int T, int D, int Bcap, int nchunk,
                int cw, float eps) {
    __shared__ __half2 s_rh[kMaxT], s_nmrh[kMaxT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int j = 8 * threadIdx.x;
    const size_t tstride = (size_t)Bcap * D;
    pdl_wait();
    pdl_launch_next();
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        for (int t = warp; t < T; t += nwarps) {
            float mean, rstd;
            merge_row_stats(stats + ((size_t)t * Bcap + b) * nchunk, nchunk, cw, D, eps, lane, mean, rstd);
            if (lane == 0) {
                s_rh[t] = __float2half2_rn(rstd);
                s_nmrh[t] = __float2half2_rn(-mean * rstd);
            }
        }
        __syncthreads();
        if (j < D) {
            const __half* zc = Z + (size_t)b * D + j;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int t0 = 0; t0 < T; t0 += TB) {
                uint4 zz[TB];
#pragma unroll
                for (int u = 0; u < TB; ++u)
                    if (t0 + u < T) zz[u] = __ldg(reinterpret_cast<const uint4*>(zc + (size_t)(t0 + u) * tstride));
                __half2 part[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) part[q] = __float2half2_rn(0.f);
#pragma unroll
                for (int u = 0; u < TB; ++u)
                    if (t0 + u < T) {
                        const __half2* h = reinterpret_cast<const __half2*>(&zz[u]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) part[q] = __hadd2(part[q], __hfma2(h[q], s_rh[t0 + u], s_nmrh[t0 + u]));
                    }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 pf = __half22float2(part[q]);
                    acc[2 * q] += pf.x;
                    acc[2 * q + 1] += pf.y;
                }
            }
            float o[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) o[u] = fmaf(g2[j + u], acc[u] / (float)T, be2[j + u]);
            float4* dst = reinterpret_cast<float4*>(pooled + (size_t)b * D + j);
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
        __syncthreads();
    }
}

}  // namespace

bool pdl_enabled() {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_PDL");
        env = (v && v[0] == '0') ? 0 : 1;
    }
    return env == 1;
}

// Launcher checks of the bounds-checked build: the sizes describe the buffers
// the kernels index (token-major [T][Bcap][D] rows, per-row chunk statistics).
cudaError_t check_mix_args(bool from_z, const MixLnArgs& a) {
    RM_HOST_BOUNDS(a.B <= a.Bcap && a.T >= 1 && a.T <= kMaxT && a.D >= 1 && a.q >= 1 && a.q * a.T == a.D);
    RM_HOST_BOUNDS(a.S != nullptr && a.g1 != nullptr && a.be1 != nullptr);
    RM_HOST_BOUNDS(from_z ? (a.Z != nullptr && a.stats != nullptr && a.g2 != nullptr && a.be2 != nullptr &&
                             a.nchunk >= 1 && a.cw >= 1 && a.nchunk * a.cw == a.D)
                          : a.X != nullptr);
    RM_HOST_BOUNDS(((reinterpret_cast<uintptr_t>(from_z ? a.Z : a.X) | reinterpret_cast<uintptr_t>(a.S)) & 15u) == 0);
    return cudaSuccess;
}

cudaError_t launch_mix_ln1(Act act, bool from_z, const MixLnArgs& a, int num_sms, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (kDebugBounds) {
        const cudaError_t e = check_mix_args(from_z, a);
        if (e != cudaSuccess) return e;
    }
    if (act == Act::BF16) {
        if (v8_ok(from_z, a)) return from_z ? launch_v8_dispatch<true>(a, num_sms, s) : launch_v8_dispatch<false>(a, num_sms, s);
        if (staged_ok(a))
            return from_z ? launch_staged_dispatch<__half, true>(a, num_sms, s)
                          : launch_staged_dispatch<__nv_bfloat16, false>(a, num_sms, s);
        return from_z ? launch_direct_dispatch<__nv_bfloat16, __half, true>(a, num_sms, s)
                      : launch_direct_dispatch<__nv_bfloat16, __half, false>(a, num_sms, s);
    }
    return from_z ? launch_direct_dispatch<float, float, true>(a, num_sms, s)
                  : launch_direct_dispatch<float, float, false>(a, num_sms, s);
}

cudaError_t launch_mix_residual_debug(bool from_z, const MixLnArgs& a, int num_sms, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    RM_HOST_BOUNDS(a.B <= a.Bcap && a.T <= kMaxT && a.q * a.T == a.D);
    if (!a.Ydbg || !v8_ok(from_z, a)) return cudaErrorNotSupported;
    return from_z ? launch_v8_dispatch<true, true>(a, num_sms, s) : launch_v8_dispatch<false, true>(a, num_sms, s);
}

cudaError_t launch_ln2_out(Act act, const void* Z, const float2* stats, const float* g2, const float* be2,
                           void* X_out, bool out_f32, int B, int T, int D, int Bcap, int nchunk, int cw, float eps,
                           int num_sms, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    RM_HOST_BOUNDS(B <= Bcap && nchunk >= 1 && nchunk * cw == D && Z != nullptr && stats != nullptr && X_out != nullptr);
    const int grid = grid_for((long long)B * T * 32, 256, num_sms * 8);
    if (act == Act::BF16 && D % 256 == 0) {
        if (out_f32)
            launch_k(ln2_out_vec_kernel<float>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, g2, be2,
                     (float*)X_out, B, T, D, Bcap, nchunk, cw, eps);
        else
            launch_k(ln2_out_vec_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, g2, be2,
                     (__nv_bfloat16*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    } else if (act == Act::BF16) {
        if (out_f32)
            launch_k(ln2_out_kernel<__half, float>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, g2, be2,
                     (float*)X_out, B, T, D, Bcap, nchunk, cw, eps);
        else
            launch_k(ln2_out_kernel<__half, __nv_bfloat16>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, g2,
                     be2, (__nv_bfloat16*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    } else {
        launch_k(ln2_out_kernel<float, float>, dim3(grid), dim3(256), 0, s, (const float*)Z, stats, g2, be2,
                 (float*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    }
    return cudaGetLastError();
}

cudaError_t launch_ln2_out_op(Act act, const void* Z, const float2* stats, int nchunk, int cw, const float* g2,
                              const float* be2, void* X_out, int B, int T, int D, int Bcap, float eps, int num_sms,
                              cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    RM_HOST_BOUNDS(B <= Bcap && nchunk >= 1 && nchunk * cw == D && Z != nullptr && stats != nullptr && X_out != nullptr);
    const int grid = grid_for((long long)B * T * 32, 256, num_sms * 8);
    if (act == Act::BF16 && D % 256 == 0)
        launch_k(ln2_out_vec_kernel<__half>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, g2, be2,
                 (__half*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    else if (act == Act::BF16)
        launch_k(ln2_out_kernel<__half, __half>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, g2, be2,
                 (__half*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    else
        launch_k(ln2_out_kernel<float, float>, dim3(grid), dim3(256), 0, s, (const float*)Z, stats, g2, be2,
                 (float*)X_out, B, T, D, Bcap, nchunk, cw, eps);
    return cudaGetLastError();
}

cudaError_t launch_pool(Act act, const void* Z, const float2* stats, const float* g2, const float* be2,
                        float* pooled, void* XL, bool xl_f32, int B, int T, int D, int Bcap, int nchunk, int cw,
                        float eps, int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (T > kMaxT) return cudaErrorNotSupported;
    RM_HOST_BOUNDS(B <= Bcap && nchunk >= 1 && nchunk * cw == D && Z != nullptr && stats != nullptr && pooled != nullptr);
    if (act == Act::BF16 && XL == nullptr && D % 8 == 0 && D <= 8 * 256) {
        int threads = (D / 8 + 31) / 32 * 32;
        if (threads < 64) threads = 64;
        const int grid = B < num_sms * 10 ? B : num_sms * 10;
        launch_k(pool_vec_kernel<kPoolBatch>, dim3(grid), dim3(threads), 0, s, (const __half*)Z, stats, g2, be2,
                 pooled, B, T, D, Bcap, nchunk, cw, eps);
        return cudaGetLastError();
    }
    const int grid = B < num_sms * 8 ? B : num_sms * 8;
    if (act == Act::BF16 && xl_f32)
        launch_k(pool_kernel<__half, float>, dim3(grid), dim3(kPoolThreads), 0, s, (const __half*)Z, stats, g2, be2,
                 pooled, (float*)XL, B, T, D, Bcap, nchunk, cw, eps);
    else if (act == Act::BF16)
        launch_k(pool_kernel<__half, __nv_bfloat16>, dim3(grid), dim3(kPoolThreads), 0, s, (const __half*)Z, stats,
                 g2, be2, pooled, (__nv_bfloat16*)XL, B, T, D, Bcap, nchunk, cw, eps);
    else
        launch_k(pool_kernel<float, float>, dim3(grid), dim3(kPoolThreads), 0, s, (const float*)Z, stats, g2, be2,
                 pooled, (float*)XL, B, T, D, Bcap, nchunk, cw, eps);
    return cudaGetLastError();
}

cudaError_t launch_stats_finalize(const float2* part, float2* out, int B, int T, int Bcap, int nchunk, int cw,
                                  int num_sms, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    RM_HOST_BOUNDS(B <= Bcap && nchunk >= 1 && cw >= 1 && part != nullptr && out != nullptr);
    launch_k(stats_finalize_kernel, dim3(grid_for((long long)B * T, 256, num_sms * 8)), dim3(256), 0, s, part, out, B,
             T, Bcap, nchunk, cw);
    return cudaGetLastError();
}

cudaError_t launch_rowstats(Act act, const void* Z, float2* stats, int B, int T, int D, int Bcap, int num_sms,
                            cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T * 32, 256, num_sms * 8);
    if (act == Act::BF16)
        launch_k(rowstats_kernel<__half>, dim3(grid), dim3(256), 0, s, (const __half*)Z, stats, B, T, D, Bcap);
    else
        launch_k(rowstats_kernel<float>, dim3(grid), dim3(256), 0, s, (const float*)Z, stats, B, T, D, Bcap);
    return cudaGetLastError();
}

cudaError_t launch_token_to_sample(Act act, const void* src, void* dst, bool out_f32, int B, int T, int D, int Bcap,
                                   cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int grid = grid_for((long long)B * T * D, 256);
    if (act == Act::BF16 && out_f32)
        token_to_sample_kernel<__half, float><<<grid, 256, 0, s>>>((const __half*)src, (float*)dst, B, T, D, Bcap);
    else if (act == Act::BF16)
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

cudaError_t launch_debug_gelu(const float* u, float* out, long long n, int form, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    debug_gelu_kernel<<<grid_for(n, 256), 256, 0, s>>>(u, out, n, form);
    return cudaGetLastError();
}

cudaError_t launch_debug_wait(const int* flag, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    debug_wait_kernel<<<1, 32, 0, s>>>(flag, err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace rm
