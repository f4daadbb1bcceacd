// Grouped fp16 GEMMs of the block backward pass on the 5th-generation tensor
// cores (sm_103a): the forward recompute of the per-token FFN, the two
// data-gradient products and the two weight-gradient products of
// "RankMixer 详解（1）" section 5.2, per token t:
//   recompute  U = S W1 + b1 (Act = Gelu(U), Gp = Gelu'(U)),  Z = Act W2 + b2 + S
//   dA = dZ W2^T  -> dU = dA * Gp                 (A = dZ, K-major; B = W2 [F][D], K-major)
//   dS = dU W1^T + dZ                             (A = dU, K-major; B = W1 [D][F], K-major)
//   dW2 = Act^T dZ,  dW1 = S^T dU                 (A and B MN-major: K is the batch)
// The recompute reads W1 [D][F] and W2 [F][D] as MN-major B operands, so a
// single fp16 copy of the weights in the pages' layout serves every product.
// dZ and dU carry a per-token power-of-two scale (see rm_train.h); the
// epilogues of the products that read them multiply by its inverse.
//
// Kernel structure (one persistent CTA per SM, 12 warps, 128 x 256 tiles):
//   warp 0      TMA producer: A and B tiles of one 64-deep k-block per stage
//               (K-major: one box of 64 x rows; MN-major: boxes of 64 x 64,
//               64 rows of the M/N dimension each) with the 128-byte swizzle
//   warp 1      MMA issuer: lane 0 issues tcgen05.mma (M = 128, N = 256, K = 16)
//               into a double-buffered TMEM accumulator
//   warp 2      TMEM allocator
//   warps 4-11  epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. 32
//               rows; the two warps of a lane quadrant split the 256 columns)
// Every mbarrier wait is bounded in time; on expiry the CTA latches an error
// word and all roles unwind.
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "rm_common.cuh"
#include "rm_train.h"
#include "rm_train_math.cuh"

namespace rm {
namespace ttc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;               // one 64-deep k-block of this CTA's 128 rows of A
constexpr int MN_BOX_BYTES = 64 * BK * 2;          // one 64 (M/N) x 64 (K) box of an MN-major operand
constexpr int TMEM_COLS = 2 * BN;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_LIMIT = 227 * 1024;
// Epilogue warps: 8 (two per TMEM lane quadrant).  16 warps for the heavy
// epilogues measured the same (2.03 against 2.05 ms for the Gelu and Gelu'
// epilogue at the 1B shape): the wait on each TMEM load was the cost, which
// loading the next 32 columns during the current ones removes.
//
// The epilogue with Gelu and Gelu' outputs stores through shared memory and
// TMA tensor stores (32 x 32 fp16 blocks, two outputs, two buffers each per
// warp, 8 KB per warp, plus the warp's 128 bias values): a lane's row of 64
// bytes is one 16-byte store per quarter instead of 32 rows' scattered
// 16-byte pieces per warp store.
//
// PAIR: a cluster of two CTAs on two SMs computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2.  CTA r loads A rows [128 r, 128 r + 128) of the
// tile and B rows (N) [128 r, 128 r + 128); the even CTA issues the MMAs
// (M = 256), which accumulate each CTA's 128 rows in its own TMEM.  A stage
// is then 32 KB per CTA instead of 48 KB, so each SM pulls a third less
// operand data from L2 per flop and more stages fit (more loads in flight).
//   full[s]   (even CTA)  1 arrival (its producer, expecting both CTAs' bytes)
//   empty[s]  (each CTA)  1 arrival: multicast commit from the even CTA
//   tfull[a]  (each CTA)  1 arrival: multicast commit from the even CTA
//   tempty[a] (even CTA)  2 x 8 arrivals: every epilogue warp of both CTAs
template <int EPI, bool PAIR>
struct KCfg {
    static constexpr int WARPS = 8;
    static constexpr int THREADS = 128 + 32 * WARPS;
    static constexpr int COLS = 256 / (WARPS / 4);      // columns of the tile per epilogue warp
    static constexpr bool TMA_OUT = EPI == TE_GELU2;
    static constexpr int TM = PAIR ? 256 : BM;          // rows of C per tile
    static constexpr int BROWS = PAIR ? BN / 2 : BN;    // rows (N) of B this CTA loads
    static constexpr int B_BYTES = BROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES = TMA_OUT ? WARPS * (4 * 2048 + 4 * COLS) : 0;
    static constexpr int FIT = (SMEM_LIMIT - 1024 - EPI_BYTES - BAR_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = FIT < 7 ? FIT : 7;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
    static_assert(2 * STAGES * 8 + 4 * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(COLS == 128, "one float4 of bias per lane in the staged epilogue");
};

struct KArgs {
    int G, M, N, K;
    int m_valid;
    int m_tiles, n_tiles;
    long long tiles;
    long long c_gpitch;
    long long c_ld;
    void* c0;
    void* c1;
    const void* r;
    const float* bias;
    const float* inv_scale;
    float* colpart;
    int colpart_rows;      // partial rows per group: ceil(M / 32)
    int um_bs, um_B;       // TE_F16T: block size and samples
    long long um_L;        // TE_F16T: values per sample
    int m_fast;            // tile order: M tiles fastest (else N tiles fastest)
    int* err;
    unsigned long long timeout_ns;
};

// Shared-memory descriptors, 128-byte swizzle (layout type 2, descriptor version 1).
// K-major: 8-row core groups 1024 bytes apart (stride byte offset); the
// leading byte offset is unused.  MN-major: each 64-element run of M (or N)
// is one 64 x 64 box (8192 bytes, leading byte offset between runs); the
// 8-row groups along K are 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// kind::f16 instruction descriptor: D f32, A and B fp16 (format 0), majors
// (bit 15: A MN-major, bit 16: B MN-major), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16_any(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tile_of(long long tile, const KArgs& a, int& g, int& mb, int& nb) {
    const long long per_group = (long long)a.m_tiles * a.n_tiles;
    g = (int)(tile / per_group);
    const int rem = (int)(tile - (long long)g * per_group);
    if (a.m_fast) {                // M tiles fastest: neighbouring CTAs share the B tile
        nb = rem / a.m_tiles;
        mb = rem - nb * a.m_tiles;
    } else {                       // N tiles fastest: neighbouring CTAs share the A tile
        mb = rem / a.n_tiles;
        nb = rem - mb * a.n_tiles;
    }
}

// Two floats to an fp16 pair, saturating at +-65504 instead of overflowing.
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(sat_f16(lo), sat_f16(hi));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// v[0..31] from 32 consecutive 16-bit values at p (64-byte aligned).  RO: the
// kernel never writes them (read through the non-coherent path); otherwise a
// plain load (the values are overwritten in place later in the same thread).
template <typename T16, bool RO = true>
__device__ __forceinline__ void load16x32(const T16* p, float (&v)[32]) {
    const uint4* r4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 rr = RO ? __ldg(r4 + j) : r4[j];
        const uint32_t w[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if constexpr (std::is_same_v<T16, __half>) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[h]));
                v[8 * j + 2 * h] = f.x;
                v[8 * j + 2 * h + 1] = f.y;
            } else {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[h]));
                v[8 * j + 2 * h] = f.x;
                v[8 * j + 2 * h + 1] = f.y;
            }
        }
    }
}

__device__ __forceinline__ void store16x32(void* dst, const uint32_t (&p)[16]) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int j = 0; j < 4; ++j) d4[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
}

// Sum of v[c] over the 32 lanes for every c, left in lane c: five exchange
// rounds, each halving the values a lane holds (31 shuffles for 32 sums).
__device__ __forceinline__ float column_sums32(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? v[i] : v[i + o];
            const float keep = upper ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// Epilogue of one warp: 32 rows (TMEM lanes) x 128 columns from n0.
// Gelu / Gelu' epilogue through shared memory: per 32-column chunk each lane
// packs its row's 32 values of each output (64 bytes) into a staging block
// with the 64-byte swizzle (16-byte piece k of row r at piece k ^ ((r >> 1) & 3)),
// and lane 0 hands both blocks to the TMA engine, which clips the rows past
// the batch.  Two pairs of blocks alternate; a pair is refilled only after the
// stores that read it have finished reading (bulk wait_group.read 1).
__device__ __forceinline__ void epilogue_gelu2_tma(const KArgs& a, const CUtensorMap* tmC0, const CUtensorMap* tmC1,
                                                   int g, int m_warp, uint32_t tbase, int n0, int lane,
                                                   uint32_t stage, uint32_t sbias, int& sbuf) {
    constexpr int NC = KCfg<TE_GELU2, false>::COLS / 32;
    const uint64_t s2 = f2_splat(a.inv_scale ? __ldg(a.inv_scale + g) : 1.0f);
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);
    uint32_t rbuf[2][32];
    tmem_ld32_nowait(tbase, rbuf[0]);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c + 1 < NC) tmem_ld32_nowait(tbase + 32u * (c + 1), rbuf[(c + 1) & 1]);
        const uint32_t* r = rbuf[c & 1];
        uint32_t pa[16], pg[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 bb = ld_shared_f4(sbias + 128u * c + 16u * j);
            uint64_t v0, g0, v1, g1;
            gelu_with_grad_x2(f2_pack(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])), s2,
                              f2_pack(bb.x, bb.y), v0, g0);
            gelu_with_grad_x2(f2_pack(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])), s2,
                              f2_pack(bb.z, bb.w), v1, g1);
            pa[2 * j] = pack_f16x2_from_f2(v0);
            pa[2 * j + 1] = pack_f16x2_from_f2(v1);
            pg[2 * j] = pack_f16x2_from_f2(g0);
            pg[2 * j + 1] = pack_f16x2_from_f2(g1);
        }
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t buf0 = stage + (uint32_t)sbuf * 4096u, buf1 = buf0 + 2048u;
        const uint32_t row0 = buf0 + (uint32_t)lane * 64u, row1 = buf1 + (uint32_t)lane * 64u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            st_shared_v4(row0 + (((uint32_t)k ^ sw) << 4), pa[4 * k], pa[4 * k + 1], pa[4 * k + 2], pa[4 * k + 3]);
            st_shared_v4(row1 + (((uint32_t)k ^ sw) << 4), pg[4 * k], pg[4 * k + 1], pg[4 * k + 2], pg[4 * k + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (m_warp < a.m_valid) {
                tma_store_3d(tmC0, buf0, n0 + 32 * c, m_warp, g);
                tma_store_3d(tmC1, buf1, n0 + 32 * c, m_warp, g);
            }
            bulk_commit_group();
        }
        sbuf ^= 1;
        if (c + 1 < NC) tmem_wait_ld();
    }
}

template <int EPI>
__device__ __forceinline__ void epilogue(const KArgs& a, int g, int m, bool valid, uint32_t tbase, int n0, int lane,
                                         int prow) {
    const size_t row = (size_t)g * (size_t)a.c_gpitch + (size_t)m * (size_t)a.c_ld + (size_t)n0;
    const float inv_s = a.inv_scale ? __ldg(a.inv_scale + g) : 1.0f;
    constexpr int NC = KCfg<EPI, false>::COLS / 32;
    // chunk c + 1 loads from TMEM while chunk c is processed (two register sets)
    uint32_t rbuf[2][32];
    tmem_ld32_nowait(tbase, rbuf[0]);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c + 1 < NC) tmem_ld32_nowait(tbase + 32u * (c + 1), rbuf[(c + 1) & 1]);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rbuf[c & 1][i]);
        const size_t off = row + 32 * c;
        if (EPI == TE_RESID) {
            if (valid) {
                const float4* b4 = reinterpret_cast<const float4*>(a.bias + (size_t)g * a.N + n0 + 32 * c);
                float rr[32];
                load16x32(reinterpret_cast<const __half*>(a.r) + off, rr);
                uint32_t p[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bb = __ldg(b4 + j);
                    p[2 * j] = f16x2_bits(fmaf(v[4 * j], inv_s, bb.x) + rr[4 * j],
                                          fmaf(v[4 * j + 1], inv_s, bb.y) + rr[4 * j + 1]);
                    p[2 * j + 1] = f16x2_bits(fmaf(v[4 * j + 2], inv_s, bb.z) + rr[4 * j + 2],
                                              fmaf(v[4 * j + 3], inv_s, bb.w) + rr[4 * j + 3]);
                }
                store16x32(reinterpret_cast<__half*>(a.c0) + off, p);
            }
        } else if (EPI == TE_DGELU) {
            if (valid) {
                float gp[32];
                load16x32<__half, false>(reinterpret_cast<const __half*>(a.r) + off, gp);
                uint32_t p[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    p[j] = f16x2_bits(v[2 * j] * gp[2 * j], v[2 * j + 1] * gp[2 * j + 1]);
                    // sum what the next products read (the stored fp16 value), unscaled
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&p[j]));
                    v[2 * j] = f.x * inv_s;
                    v[2 * j + 1] = f.y * inv_s;
                }
                store16x32(reinterpret_cast<__half*>(a.c0) + off, p);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            const float s = column_sums32(v, lane);
            a.colpart[((size_t)g * a.colpart_rows + prow) * a.N + n0 + 32 * c + lane] = s;
        } else if (EPI == TE_DRESID) {
            if (valid) {
                const float4* r4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.r) + off);
                float4* d4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.c0) + off);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 rr = __ldg(r4 + j);
                    d4[j] = make_float4(fmaf(v[4 * j], inv_s, rr.x), fmaf(v[4 * j + 1], inv_s, rr.y),
                                        fmaf(v[4 * j + 2], inv_s, rr.z), fmaf(v[4 * j + 3], inv_s, rr.w));
                }
            }
        } else if (EPI == TE_BIAS_IO) {       // bf16 output (tensor-core path: bf16 contexts)
            if (valid) {
                const float4* b4 = reinterpret_cast<const float4*>(a.bias + (size_t)g * a.N + n0 + 32 * c);
                uint32_t p[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bb = __ldg(b4 + j);
                    const __nv_bfloat162 h0 = __floats2bfloat162_rn(v[4 * j] + bb.x, v[4 * j + 1] + bb.y);
                    const __nv_bfloat162 h1 = __floats2bfloat162_rn(v[4 * j + 2] + bb.z, v[4 * j + 3] + bb.w);
                    p[2 * j] = *reinterpret_cast<const uint32_t*>(&h0);
                    p[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&h1);
                }
                store16x32(reinterpret_cast<__nv_bfloat16*>(a.c0) + off, p);
            }
        } else if (EPI == TE_F16T) {
            // column n = b bs + r of row m -> Y[b][m bs + r]: 8-column groups never
            // straddle samples (bs % 8 == 0), each one 16-byte store
            if (valid) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int n = n0 + 32 * c + 8 * q;
                    const int b = n / a.um_bs;
                    if (b < a.um_B) {
                        const int r = n - b * a.um_bs;
                        uint4 w;
                        w.x = f16x2_bits(v[8 * q] * inv_s, v[8 * q + 1] * inv_s);
                        w.y = f16x2_bits(v[8 * q + 2] * inv_s, v[8 * q + 3] * inv_s);
                        w.z = f16x2_bits(v[8 * q + 4] * inv_s, v[8 * q + 5] * inv_s);
                        w.w = f16x2_bits(v[8 * q + 6] * inv_s, v[8 * q + 7] * inv_s);
                        *reinterpret_cast<uint4*>(reinterpret_cast<__half*>(a.c0) + (size_t)b * a.um_L +
                                                  (size_t)m * a.um_bs + r) = w;
                    }
                }
            }
        } else if (EPI == TE_F16) {
            if (valid) {
                uint32_t p[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) p[j] = f16x2_bits(v[2 * j] * inv_s, v[2 * j + 1] * inv_s);
                store16x32(reinterpret_cast<__half*>(a.c0) + off, p);
            }
        } else {   // TE_F32
            if (valid) {
                float4* d4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.c0) + off);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    d4[j] = make_float4(v[4 * j] * inv_s, v[4 * j + 1] * inv_s, v[4 * j + 2] * inv_s,
                                        v[4 * j + 3] * inv_s);
            }
        }
        if (c + 1 < NC) tmem_wait_ld();
    }
}

template <int EPI, bool A_MN, bool B_MN, bool PAIR>
__global__ void __launch_bounds__(KCfg<EPI, PAIR>::THREADS, 1)
train_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                     const KArgs args) {
    using C = KCfg<EPI, PAIR>;
    constexpr int STAGES = C::STAGES;
    constexpr int STAGE_BYTES = C::STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * A_BYTES;
    const uint32_t sEpi = base + STAGES * STAGE_BYTES;                 // TMA-store staging (1024-aligned)
    const uint32_t bar0 = sEpi + C::EPI_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int x) { return bar0 + 8u * (2 * STAGES + x); };
    auto tempty_bar = [&](int x) { return bar0 + 8u * (2 * STAGES + 2 + x); };
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + STAGES * STAGE_BYTES + C::EPI_BYTES + 8 * (2 * STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;    // 0: issues the MMAs
    const long long unit = PAIR ? (long long)(blockIdx.x >> 1) : (long long)blockIdx.x;
    const long long nunits = PAIR ? (long long)(gridDim.x >> 1) : (long long)gridDim.x;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(tfull_bar(x), 1);
            mbar_init(tempty_bar(x), PAIR ? 2 * C::WARPS : C::WARPS * 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();    // both CTAs' barriers and TMEM exist before any cross-CTA use
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
    const int kblocks = (args.K + BK - 1) / BK;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long tile = unit; ok && tile < args.tiles; tile += nunits) {
            int g, mb, nb;
            tile_of(tile, args, g, mb, nb);
            const int arow = mb * C::TM + BM * (int)rank;
            const int brow = nb * BN + C::BROWS * (int)rank;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, args.err, args.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    // the even CTA's full barrier counts both CTAs' bytes
                    const uint32_t fb = PAIR ? mapa_shared(full_bar(stage), 0) : full_bar(stage);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), (uint32_t)((PAIR ? 2 : 1) * STAGE_BYTES));
                    const uint32_t a_dst = sA + stage * A_BYTES;
                    const uint32_t b_dst = sB + stage * C::B_BYTES;
                    auto load = [&](const CUtensorMap* m, uint32_t dst, int x, int y) {
                        if constexpr (PAIR)
                            tma_load_3d_pair(m, dst, fb, x, y, g);
                        else
                            tma_load_3d(m, dst, fb, x, y, g);
                    };
                    if (A_MN) {
#pragma unroll
                        for (int i = 0; i < BM / 64; ++i) load(&tmA, a_dst + i * MN_BOX_BYTES, arow + 64 * i, kb * BK);
                    } else {
                        load(&tmA, a_dst, kb * BK, arow);
                    }
                    if (B_MN) {
#pragma unroll
                        for (int i = 0; i < C::BROWS / 64; ++i)
                            load(&tmB, b_dst + i * MN_BOX_BYTES, brow + 64 * i, kb * BK);
                    } else {
                        load(&tmB, b_dst, kb * BK, brow);
                    }
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1 && rank == 0) {
        // ------------------------------ MMA issuer --------------------------------
        constexpr uint32_t idesc = idesc_f16(C::TM, BN, A_MN, B_MN);
        // per 16-deep step: K-major operands advance 32 bytes inside the swizzled
        // row, MN-major operands 16 rows of 128 bytes
        constexpr uint32_t a_step = A_MN ? 2048u : 32u, b_step = B_MN ? 2048u : 32u;
        constexpr uint32_t a_lbo = A_MN ? (uint32_t)MN_BOX_BYTES : 16u, b_lbo = B_MN ? (uint32_t)MN_BOX_BYTES : 16u;
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (long long tile = unit; ok && tile < args.tiles; tile += nunits) {
            if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err, args.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.err, args.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sA + stage * A_BYTES;
                const uint32_t b0 = sB + stage * C::B_BYTES;
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = sw128_desc(a0 + a_step * k, a_lbo, 1024u);
                        const uint64_t bd = sw128_desc(b0 + b_step * k, b_lbo, 1024u);
                        if constexpr (PAIR)
                            umma_f16_pair(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                        else
                            umma_f16_any(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    if constexpr (PAIR)
                        umma_commit_pair_mc(empty_bar(stage), (uint16_t)0x3);
                    else
                        umma_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (lane == 0) {
                if constexpr (PAIR)
                    umma_commit_pair_mc(tfull_bar(acc), (uint16_t)0x3);
                else
                    umma_commit(tfull_bar(acc));
            }
            __syncwarp();
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    } else if (warp >= 4) {
        // ------------------------------ epilogue ----------------------------------
        const int ew = warp - 4;
        const int quad = warp & 3;
        const int half = ew >> 2;               // which group of C::COLS columns
        const uint32_t stage = sEpi + (uint32_t)ew * 8192u;
        const uint32_t sbias = sEpi + (uint32_t)C::WARPS * 8192u + (uint32_t)ew * (4u * C::COLS);
        int sbuf = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (long long tile = unit; tile < args.tiles; tile += nunits) {
            int g, mb, nb;
            tile_of(tile, args, g, mb, nb);
            float4 bias4;
            if constexpr (C::TMA_OUT)     // this warp's bias slice, loaded during the wait
                bias4 = __ldg(reinterpret_cast<const float4*>(args.bias + (size_t)g * args.N + nb * BN +
                                                              half * C::COLS) + lane);
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.err, args.timeout_ns)) break;
            tc_fence_after();
            if constexpr (C::TMA_OUT) {
                __syncwarp();                           // the previous tile's reads of the slice are done
                st_shared_v4(sbias + 16u * lane, __float_as_uint(bias4.x), __float_as_uint(bias4.y),
                             __float_as_uint(bias4.z), __float_as_uint(bias4.w));
                __syncwarp();
            }
            const int m = mb * C::TM + BM * (int)rank + quad * 32 + lane;
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN + half * C::COLS);
            if constexpr (C::TMA_OUT)
                epilogue_gelu2_tma(args, &tmC0, &tmC1, g, m - lane, tbase, nb * BN + half * C::COLS, lane, stage,
                                   sbias, sbuf);
            else
                epilogue<EPI>(args, g, m, m < args.m_valid, tbase, nb * BN + half * C::COLS, lane,
                              (mb * C::TM + BM * (int)rank) / kTrainColpartRows + quad);
            tc_fence_before();
            if constexpr (PAIR) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            } else {
                mbar_arrive(tempty_bar(acc));
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (C::TMA_OUT && lane == 0) bulk_wait_group<0>();   // this warp's tensor stores have landed
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();    // no CTA leaves while its peer may still touch its memory
    if (warp == 2) {
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

// 3-D fp16 map {inner, outer, G} with the given box (inner box 64 = 128 bytes).
bool make_map(CUtensorMap* m, const TOperand& op, int G, int box_outer) {
    if (!get_encoder()) return false;
    cuuint64_t dims[3] = {(cuuint64_t)op.inner, (cuuint64_t)op.outer, (cuuint64_t)G};
    cuuint64_t strides[2] = {(cuuint64_t)(op.ld ? op.ld : op.inner) * 2, (cuuint64_t)op.gpitch * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_outer, 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 output map over [G][rows][N] (row pitch ld, group pitch gpitch): box
// 32 x 32 x 1 with the 64-byte swizzle; rows at or past `rows` are clipped.
bool make_map_out(CUtensorMap* m, void* ptr, int N, int rows, int G, long long ld, long long gpitch) {
    if (!get_encoder()) return false;
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)rows, (cuuint64_t)G};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)gpitch * 2};
    cuuint32_t box[3] = {32u, 32u, 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, ptr, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, bool A_MN, bool B_MN, bool PAIR>
cudaError_t run(const TrainGemm& g, const KArgs& ka, int num_sms, cudaStream_t s) {
    using C = KCfg<EPI, PAIR>;
    CUtensorMap mA, mB, mC0, mC1;
    if (!make_map(&mA, g.a, g.G, A_MN ? BK : BM)) return cudaErrorInvalidValue;
    if (!make_map(&mB, g.b, g.G, B_MN ? BK : C::BROWS)) return cudaErrorInvalidValue;
    if constexpr (C::TMA_OUT) {
        if (!make_map_out(&mC0, g.c0, g.N, g.m_valid, g.G, ka.c_ld, g.c_gpitch)) return cudaErrorInvalidValue;
        if (!make_map_out(&mC1, g.c1, g.N, g.m_valid, g.G, ka.c_ld, g.c_gpitch)) return cudaErrorInvalidValue;
    } else {
        mC0 = mA;   // unused
        mC1 = mA;
    }
    auto k = train_gemm_tc_kernel<EPI, A_MN, B_MN, PAIR>;
    constexpr int smem = C::SMEM_BYTES;
    {
        cudaError_t e = smem_attr_once((const void*)k, smem);
        if (e != cudaSuccess) return e;
    }
    // persistent: one CTA (or CTA pair) per SM (pair of SMs), at most one per tile
    const long long units = PAIR ? num_sms / 2 : num_sms;
    const long long grid = (ka.tiles < units ? ka.tiles : units) * (PAIR ? 2 : 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, mA, mB, mC0, mC1, ka);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// CTA pairs where they measured faster at the 1B shape (B = 4096, per-launch
// device time): the weight gradients, both operands MN-major with six TMA
// boxes per single-CTA stage (1658 -> 1595 us), and the Gelu / Gelu' product,
// whose epilogue staging leaves a single CTA only 3 stages (about 1.84 ->
// 1.71 ms), and UniMixing's global product (16 k-blocks per tile: 522 -> 339
// us).  The other products ran slower as pairs (Z 1406 -> 1539 us, dU
// 1756 -> 1815, dS 1529 -> 1606) and keep one CTA per tile.  Pairs need at
// least two 128-row blocks (and whole 256-row tiles of an MN-major A).
bool use_pair(int epi, const TrainGemm& g, int num_sms) {
    const bool wanted = epi == TE_GELU2 || epi == TE_F16T || (epi == TE_F32 && g.a.mn && g.b.mn);
    return wanted && num_sms >= 2 && g.m_valid > BM && (!g.a.mn || g.M % (2 * BM) == 0);
}

}  // namespace ttc

bool train_tc_supported(const TrainGemm& g) {
    auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (g.N % ttc::BN != 0 || g.M < 1 || g.K < 1 || g.G < 1) return false;
    if (!aligned(g.a.ptr) || !aligned(g.b.ptr)) return false;
    if ((g.c0 && !aligned(g.c0)) || (g.c1 && !aligned(g.c1))) return false;   // TMA stores, 16-byte vectors
    // K-major operands: K is the inner extent and must fill whole 64-deep k-blocks
    if (!g.a.mn && (g.a.inner != g.K || g.K % ttc::BK != 0)) return false;
    if (!g.b.mn && (g.b.inner != g.K || g.K % ttc::BK != 0)) return false;
    // MN-major operands: whole 128-row (A) / 256-column (B) tiles of the inner extent
    if (g.a.mn && (g.a.inner != g.M || g.M % ttc::BM != 0)) return false;
    if (g.b.mn && (g.b.inner != g.N)) return false;
    if (g.a.gpitch % 8 != 0 || g.b.gpitch % 8 != 0) return false;
    if (g.a.ld % 8 != 0 || g.b.ld % 8 != 0) return false;         // 16-byte row pitches for TMA
    if ((g.c_ld ? g.c_ld : g.N) % 8 != 0 || g.c_gpitch % 8 != 0) return false;   // 16-byte vector stores
    if (g.um_bs % 8 != 0 || g.um_L % 8 != 0) return false;   // TE_F16T: 8-column groups inside one sample
    return true;
}

int train_colpart_rows(const TrainGemm& g, int num_sms) {
    const int tm = ttc::use_pair(TE_DGELU, g, num_sms) ? 2 * ttc::BM : ttc::BM;
    return (g.m_valid + tm - 1) / tm * (tm / kTrainColpartRows);
}

cudaError_t launch_train_gemm_tc(int epi, const TrainGemm& g, int num_sms, cudaStream_t s) {
    if (!train_tc_supported(g)) return cudaErrorNotSupported;
    const bool pair = ttc::use_pair(epi, g, num_sms);
    const int tm = pair ? 2 * ttc::BM : ttc::BM;
    ttc::KArgs ka{};
    ka.G = g.G;
    ka.M = g.M;
    ka.N = g.N;
    ka.K = g.K;
    ka.m_valid = g.m_valid;
    ka.m_tiles = (g.m_valid + tm - 1) / tm;
    ka.n_tiles = g.N / ttc::BN;
    ka.tiles = (long long)g.G * ka.m_tiles * ka.n_tiles;
    ka.c_gpitch = g.c_gpitch;
    ka.c_ld = g.c_ld ? g.c_ld : g.N;
    ka.c0 = g.c0;
    ka.c1 = g.c1;
    ka.r = g.r;
    ka.bias = g.bias;
    ka.inv_scale = g.inv_scale;
    ka.colpart = g.colpart;
    ka.um_bs = g.um_bs;
    ka.um_B = g.um_B;
    ka.um_L = g.um_L;
    // Tile order.  N tiles fastest re-reads a group's whole B operand once per M
    // tile, which costs DRAM traffic only when B outgrows L2; then walk M fastest
    // if A is the smaller operand (UniMixing's global product: A 2 MB, B 403 MB
    // at the 1B shape read 4x from DRAM in N order).  Every other product here has
    // per-group operands within L2 and keeps N order.
    {
        const double a_bytes = 2.0 * (double)g.m_valid * g.K, b_bytes = 2.0 * (double)g.N * g.K;
        ka.m_fast = (b_bytes > 64.0 * 1024 * 1024 && a_bytes < b_bytes && ka.m_tiles > 1) ? 1 : 0;
    }
    ka.colpart_rows = train_colpart_rows(g, num_sms);
    ka.err = g.err;
    ka.timeout_ns = g.timeout_ns;
    if (ka.tiles == 0) return cudaSuccess;
    const bool amn = g.a.mn, bmn = g.b.mn;
#define RM_TRAIN_RUN(E, AMN, BMN) \
    return pair ? ttc::run<E, AMN, BMN, true>(g, ka, num_sms, s) : ttc::run<E, AMN, BMN, false>(g, ka, num_sms, s)
    switch (epi) {
        case TE_GELU2:
            if (!amn && bmn) RM_TRAIN_RUN(TE_GELU2, false, true);
            break;
        case TE_RESID:
            if (!amn && bmn) RM_TRAIN_RUN(TE_RESID, false, true);
            break;
        case TE_DGELU:
            if (!amn && !bmn) RM_TRAIN_RUN(TE_DGELU, false, false);
            break;
        case TE_DRESID:
            if (!amn && !bmn) RM_TRAIN_RUN(TE_DRESID, false, false);
            break;
        case TE_F32:
            if (amn && bmn) RM_TRAIN_RUN(TE_F32, true, true);
            if (!amn && !bmn) RM_TRAIN_RUN(TE_F32, false, false);
            break;
        case TE_BIAS_IO:
            if (!amn && bmn) RM_TRAIN_RUN(TE_BIAS_IO, false, true);
            break;
        case TE_F16:
            if (!amn && bmn) RM_TRAIN_RUN(TE_F16, false, true);
            break;
        case TE_F16T:
            if (!amn && bmn && g.um_bs % 8 == 0 && g.um_bs > 0) RM_TRAIN_RUN(TE_F16T, false, true);
            break;
        default: break;
    }
#undef RM_TRAIN_RUN
    return cudaErrorNotSupported;
}

}  // namespace rm
