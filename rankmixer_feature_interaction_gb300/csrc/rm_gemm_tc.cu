// Grouped per-token FFN GEMMs on the 5th-generation tensor cores (sm_103a).
//
// "RankMixer: Scaling Up Ranking Models in Industrial Recommenders", section
// 3.3.2 Eq. 6-9: token t owns W1_t (D x kD) and W2_t (kD x D).  The same-
// position rows of a batch form a B x D matrix multiplied by that token's
// weights ("RankMixer 详解（1）" section 4.3), so a layer's PFFN is T
// independent GEMMs of equal shape -- one group per token.
//
//   GEMM1: Hid[t] = Gelu(S[t] W1_t + b1_t)            (M = B, N = kD, K = D)
//   GEMM2: Z[t]   = Hid[t] W2_t + b2_t + S[t]         (M = B, N = D,  K = kD)
//          stored in fp16, plus per-row, per-chunk LayerNorm partials
//          (mean, M2) of the float32 values
// Operands are fp16 (10-bit mantissa; the weights are converted exactly from
// bf16 when the context is created), accumulation is fp32 in TMEM.
//
// Kernel structure (one persistent CTA per SM, 12 warps):
//   warp 0      TMA producer: 128x64 A and BNx64 B tiles (128-byte swizzle)
//               into a STAGES-deep shared-memory ring, completion counted on
//               "full" mbarriers
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16)
//               into a double-buffered TMEM accumulator, frees ring slots with
//               tcgen05.commit on the "empty" mbarriers
//   warp 2      TMEM allocator
//   warps 4-11  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31, i.e. tile rows; two warps per lane
//               quadrant split the columns), fused bias + GELU (GEMM1) or
//               bias + residual + row statistics (GEMM2), global stores
// Every mbarrier wait is bounded in time; on expiry the CTA latches an error
// word, the other roles see an abort flag and all of them unwind.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "rm_common.cuh"
#include "rm_internal.h"

namespace rm {

cudaError_t smem_attr_once(const void* func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> done;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(func, dev);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

int pair_occupancy_once(const void* func, int threads, int smem, int num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return num_sms / 2;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(func, dev);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * (num_sms / 2)), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = num_sms / 2;
    }
    cache[key] = n;
    return n;
}

namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                 // one 128-byte swizzle row of fp16
constexpr int kEpiWarps = 8;
constexpr int kThreads = 128 + kEpiWarps * 32;

enum { EPI_GELU = 1, EPI_RESID = 2, EPI_GATED = 3 };

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    static constexpr int EPI_BYTES = kEpiWarps * 2 * 2048;   // per epilogue warp: two 32 x 32 fp16 blocks
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr int COLS_PER_WARP = BN / 2;        // two epilogue warps per lane quadrant
    static constexpr int CHUNKS = COLS_PER_WARP / 32;
    static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation must be a power of 2");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(CHUNKS >= 1, "BN >= 64");
    static_assert(2 * STAGES * 8 + 4 * 8 + 8 <= BAR_BYTES, "barrier area");
};

struct Args {
    int N, K;
    int ngroups;              // groups in this launch
    int group_base, group_stride;   // weight group of launch group j: group_base + j * group_stride
    // uniform groups (dense PFFN): M rows each, A rows of group j start at j * a_group_rows
    int M;
    long long a_group_rows;
    int m_tiles;              // ceil(M / BM), uniform groups only
    int n_tiles;
    int n_fastest;            // uniform groups: walk N tiles fastest (A tile shared by neighbours)
    long long tiles;          // uniform groups only
    // variable groups (MoE experts), indexed by weight group: row count and first packed row;
    // tile_prefix[j] = sum over launch groups i < j of ceil(count / BM)  (length ngroups + 1)
    const int* g_count;
    const int* g_off;
    const int* tile_prefix;
    const float* bias;        // [weight groups][N]
    __half* hid;              // EPI_GELU output rows (same row index as A), fp16
    int hid_tma;              // EPI_GELU, uniform groups: store through shared memory with TMA (output map)
    int hid_evict_first;      // hid_tma: the tensor stores carry the L2 evict-first hint
    long long rows_cap;       // rows of the output, residual and statistics buffers (bounds-checked build)
    const __half* resid;      // EPI_RESID residual rows (same row index as A), fp16
    __half* z;                // EPI_RESID output rows (fp16)
    float2* stats;            // EPI_RESID row partials [row][nchunk]
    int nchunk;
    const float* row_gate;    // EPI_GATED: gate of each packed row (same row index as A)
    int* err;
    unsigned long long timeout_ns;
};

// Tiled TMA store whose lines L2 evicts first: written rows that no later
// work of the launch reads soon (a hidden layer larger than L2) then push out
// fewer of the operand tiles that neighbouring CTAs still re-read.
__device__ __forceinline__ void tma_store_3d_evict_first(const CUtensorMap* m, uint32_t src, int x, int y, int z) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], pol;\n\t}"
        ::"l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// v[0..31] += 32 consecutive fp16 values at p (64-byte aligned).
__device__ __forceinline__ void add_f16x32(float (&v)[32], const __half* p) {
    const uint4* r4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 rr = __ldg(r4 + j);
        const uint32_t w[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const __half2 pr = *reinterpret_cast<const __half2*>(&w[h]);
            v[8 * j + 2 * h] += __low2float(pr);
            v[8 * j + 2 * h + 1] += __high2float(pr);
        }
    }
}

struct TileCoord {
    int j, mb, nb, wg, Mg;
    long long row0;           // first A row of the group
};

__device__ __forceinline__ TileCoord decode_tile(long long tile, const Args& a) {
    TileCoord c;
    if (a.tile_prefix == nullptr) {
        const long long per_group = (long long)a.m_tiles * a.n_tiles;
        c.j = (int)(tile / per_group);
        const int rem = (int)(tile - (long long)c.j * per_group);
        if (a.n_fastest) {        // neighbouring CTAs share the activation tile
            c.mb = rem / a.n_tiles;
            c.nb = rem - c.mb * a.n_tiles;
        } else {                  // neighbouring CTAs share the weight tile
            c.nb = rem / a.m_tiles;
            c.mb = rem - c.nb * a.m_tiles;
        }
        c.wg = a.group_base + c.j * a.group_stride;
        c.Mg = a.M;
        c.row0 = (long long)c.j * a.a_group_rows;
    } else {
        // largest j with tile_prefix[j] * n_tiles <= tile (skips empty groups)
        int lo = 0, hi = a.ngroups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)__ldg(a.tile_prefix + mid) * a.n_tiles <= tile) lo = mid; else hi = mid - 1;
        }
        c.j = lo;
        const int p0 = __ldg(a.tile_prefix + lo);
        const int mt = __ldg(a.tile_prefix + lo + 1) - p0;
        const int rem = (int)(tile - (long long)p0 * a.n_tiles);
        c.nb = rem / mt;
        c.mb = rem - c.nb * mt;
        c.wg = a.group_base + c.j * a.group_stride;
        c.Mg = __ldg(a.g_count + c.wg);
        c.row0 = __ldg(a.g_off + c.wg);
    }
    return c;
}

// EPI_GELU epilogue through shared memory and TMA tensor stores (uniform
// groups).  The warp's 32 rows x COLS columns are written in 32 x 32 blocks:
// each lane packs its row's 32 GELU outputs (64 bytes) into a staging block
// with the 64-byte swizzle (16-byte chunk k of row r at chunk k ^ ((r >> 1) & 3)),
// and lane 0 hands the block to the TMA engine, which writes whole lines and
// clips rows past the token group's batch.  Two staging blocks per warp
// alternate; a block is refilled only after the store that read it has
// finished reading (bulk wait_group.read 1).
template <int COLS, bool PREFETCH>
__device__ __forceinline__ void epilogue_gelu_tma(const Args& args, const TileCoord& tc, const CUtensorMap* tmC,
                                                  uint32_t tbase, int n0, int m_warp, uint32_t stage, int lane,
                                                  int& sbuf) {
    constexpr int NC = COLS / 32;
    const float* bias = args.bias + (size_t)tc.wg * args.N + n0;
    const bool any_valid = m_warp < tc.Mg;
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);
    // PREFETCH: TMEM loads run one chunk ahead, chunk c + 1 in flight while
    // chunk c is turned into GELU outputs (two register sets).  Without it
    // (more epilogue warps, fewer registers each) other warps hide the load.
    uint32_t r[PREFETCH ? 2 : 1][32];
    tmem_ld32_nowait(tbase, r[0]);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        __syncwarp();
        if (PREFETCH && c + 1 < NC) tmem_ld32_nowait(tbase + 32u * (c + 1), r[(c + 1) % (PREFETCH ? 2 : 1)]);
        if (!PREFETCH && c > 0) {
            tmem_ld32_nowait(tbase + 32u * c, r[0]);
            tmem_wait_ld();
        }
        const uint32_t* v = r[c % (PREFETCH ? 2 : 1)];
        uint32_t p[16];
        const float4* b4 = reinterpret_cast<const float4*>(bias + 32 * c);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 bb = __ldg(b4 + j);
            p[2 * j] = pack_f16x2_from_f2(gelu_erf_x2(f2_pack(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1])),
                                                      f2_pack(bb.x, bb.y)));
            p[2 * j + 1] = pack_f16x2_from_f2(
                gelu_erf_x2(f2_pack(__uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])), f2_pack(bb.z, bb.w)));
        }
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t buf = stage + (uint32_t)sbuf * 2048u;
        const uint32_t row = buf + (uint32_t)lane * 64u;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            st_shared_v4(row + (((uint32_t)k ^ sw) << 4), p[4 * k], p[4 * k + 1], p[4 * k + 2], p[4 * k + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (any_valid) {
                if (args.hid_evict_first)
                    tma_store_3d_evict_first(tmC, buf, n0 + 32 * c, m_warp, tc.j);
                else
                    tma_store_3d(tmC, buf, n0 + 32 * c, m_warp, tc.j);
            }
            bulk_commit_group();
        }
        sbuf ^= 1;
        if (PREFETCH && c + 1 < NC) tmem_wait_ld();
    }
}

// Epilogue of one accumulator tile for one warp: the warp owns 32 rows of the
// tile (its TMEM lane quadrant) and COLS columns starting at n0; `tbase` is
// the TMEM address of its first column.  Every lane takes part in the TMEM
// loads; only rows inside the group (valid) are stored.
template <int COLS, int EPI>
__device__ __forceinline__ void epilogue_tile(const Args& args, const TileCoord& tc, bool valid, long long arow,
                                              uint32_t tbase, int n0) {
    // bounds-checked build: a row inside the group must lie inside the buffers
    if (valid && !RM_IN_BOUNDS(arow >= 0 && arow < args.rows_cap && n0 + COLS <= args.N, args.err)) valid = false;
    const size_t orow = (size_t)arow * (size_t)args.N + n0;
    const float* bias = args.bias + (size_t)tc.wg * args.N + n0;
    if (EPI == EPI_GELU) {
#pragma unroll 1
        for (int c = 0; c < (COLS / 32); ++c) {
            float v[32];
            tmem_ld32(tbase + 32u * c, v);
            if (valid) {
                uint32_t p[16];
                const float4* b4 = reinterpret_cast<const float4*>(bias + 32 * c);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bb = __ldg(b4 + j);
                    p[2 * j] = pack_f16x2_from_f2(gelu_erf_x2(f2_pack(v[4 * j], v[4 * j + 1]), f2_pack(bb.x, bb.y)));
                    p[2 * j + 1] =
                        pack_f16x2_from_f2(gelu_erf_x2(f2_pack(v[4 * j + 2], v[4 * j + 3]), f2_pack(bb.z, bb.w)));
                }
                uint4* dst = reinterpret_cast<uint4*>(args.hid + orow + 32 * c);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
            }
        }
    } else if (EPI == EPI_RESID) {
        float shift = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll 1
        for (int c = 0; c < (COLS / 32); ++c) {
            float v[32];
            tmem_ld32(tbase + 32u * c, v);
            if (valid) {
                const float4* b4 = reinterpret_cast<const float4*>(bias + 32 * c);
                add_f16x32(v, args.resid + orow + 32 * c);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bb = __ldg(b4 + j);
                    v[4 * j] += bb.x;
                    v[4 * j + 1] += bb.y;
                    v[4 * j + 2] += bb.z;
                    v[4 * j + 3] += bb.w;
                }
                if (c == 0) {
                    float mm = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) mm += v[j];
                    shift = mm * (1.0f / 32.0f);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float d = v[j] - shift;
                    s1 += d;
                    s2 = fmaf(d, d, s2);
                }
                uint4* dst = reinterpret_cast<uint4*>(args.z + orow + 32 * c);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_uint4(pack_f16x2(v[8 * j], v[8 * j + 1]), pack_f16x2(v[8 * j + 2], v[8 * j + 3]),
                                        pack_f16x2(v[8 * j + 4], v[8 * j + 5]),
                                        pack_f16x2(v[8 * j + 6], v[8 * j + 7]));
            }
        }
        if (valid) {
            const float n = (float)COLS;
            const float mean = shift + s1 / n;
            const float m2 = fmaxf(s2 - s1 * s1 / n, 0.f);
            const int chunk = n0 / COLS;
            args.stats[(size_t)arow * args.nchunk + chunk] = make_float2(mean, m2);
        }
    } else {  // EPI_GATED: Y[row] = gate * (acc + b2) in fp16, row = the packed row of A
        const float gate = valid ? __ldg(args.row_gate + arow) : 0.f;
#pragma unroll 1
        for (int c = 0; c < (COLS / 32); ++c) {
            float v[32];
            tmem_ld32(tbase + 32u * c, v);
            if (valid) {
                const float4* b4 = reinterpret_cast<const float4*>(bias + 32 * c);
                uint32_t p[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bb = __ldg(b4 + j);
                    p[2 * j] = pack_f16x2(gate * (v[4 * j] + bb.x), gate * (v[4 * j + 1] + bb.y));
                    p[2 * j + 1] = pack_f16x2(gate * (v[4 * j + 2] + bb.z), gate * (v[4 * j + 3] + bb.w));
                }
                uint4* dst = reinterpret_cast<uint4*>(args.hid + orow + 32 * c);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
            }
        }
    }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
pffn_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const Args args) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sA = base;
    const uint32_t sB = base + C::STAGES * C::A_BYTES;
    const uint32_t sEpi = base + C::STAGES * C::STAGE_BYTES;           // epilogue staging, 1024-aligned
    const uint32_t bar0 = sEpi + C::EPI_BYTES;
    // barrier addresses: full[s], empty[s], tfull[2], tempty[2]
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES + 8 * (2 * C::STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiWarps * 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
    pdl_wait();              // operands and outputs are shared with the previous kernels of the stream
    pdl_launch_next();

    const int kblocks = args.K / BK;
    const long long tiles =
        args.tile_prefix ? (long long)__ldg(args.tile_prefix + args.ngroups) * args.n_tiles : args.tiles;

    // The producer and MMA warps run their loops converged (every lane waits
    // on the barriers); lane 0 issues the copies, the MMAs and their commits
    // (a commit tracks the MMAs of the thread that issues it).
    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (long long tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
                const TileCoord tc = decode_tile(tile, args);
                // A: uniform groups through a [groups][M][K] map (rows past M of a group
                // read as zeros without a memory access); variable groups as packed rows
                const int arow = args.tile_prefix ? (int)(tc.row0 + (long long)tc.mb * BM) : tc.mb * BM;
                const int agrp = args.tile_prefix ? 0 : tc.j;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, args.err, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full_bar(stage), (uint32_t)C::STAGE_BYTES);
                        tma_load_3d(&tmA, sA + stage * C::A_BYTES, full_bar(stage), kb * BK, arow, agrp);
                        tma_load_3d(&tmB, sB + stage * C::B_BYTES, full_bar(stage), kb * BK, tc.nb * BN, tc.wg);
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        {
            constexpr uint32_t idesc = make_idesc_f16_f32(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (long long tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
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
                    const uint32_t a0 = sA + stage * C::A_BYTES;
                    const uint32_t b0 = sB + stage * C::B_BYTES;
                    if (lane == 0) {
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            umma_f16(d_tmem, make_sw128_desc(a0 + 32u * k), make_sw128_desc(b0 + 32u * k), idesc,
                                     (kb > 0 || k > 0) ? 1u : 0u);
                        }
                        umma_commit(empty_bar(stage));
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) umma_commit(tfull_bar(acc));
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else if (warp >= 4) {
        // ------------------------------ epilogue ----------------------------------
        const int ew = warp - 4;
        const int quad = warp & 3;              // TMEM lanes this warp may read
        const int half = ew >> 2;               // which BN/2 columns
        const int row_in_tile = quad * 32 + lane;
        const uint32_t stage = sEpi + (uint32_t)ew * 4096u;
        int sbuf = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
            const TileCoord tc = decode_tile(tile, args);
            // every lane waits (the warp stays converged for tcgen05.ld)
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.err, args.timeout_ns)) break;
            tc_fence_after();
            const int m = tc.mb * BM + row_in_tile;          // row inside the group
            const bool valid = m < tc.Mg;
            const long long arow = tc.row0 + m;             // row of A and of the row-aligned outputs
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN + half * C::COLS_PER_WARP);
            const int n0 = tc.nb * BN + half * C::COLS_PER_WARP;
            if (EPI == EPI_GELU && args.hid_tma)
                epilogue_gelu_tma<C::COLS_PER_WARP, true>(args, tc, &tmC, tbase, n0, m - lane, stage, lane, sbuf);
            else
                epilogue_tile<C::COLS_PER_WARP, EPI>(args, tc, valid, arow, tbase, n0);
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_group<0>();   // this warp's tensor stores have landed
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}


// ----------------------------------------------------------------------------
// CTA-pair variant for the dense PFFN (uniform groups): a cluster of 2 CTAs
// on two SMs computes a 256 x BN tile with tcgen05.mma.cta_group::2.  CTA r
// of the pair loads A rows [128 r, 128 r + 128) of the tile and B rows
// [BN/2 r, BN/2 r + BN/2) into its own shared memory; the even CTA issues the
// pair MMA (M = 256), which reads both CTAs' tiles and accumulates each CTA's
// 128 rows x BN columns in that CTA's TMEM.  Per CTA a stage is 32 KB (A 16 KB
// + half of B 16 KB), so 6 stages fit and each SM pulls a third less operand
// data from L2 than the single-CTA kernel.
//   full[s]   (even CTA)  1 arrival (its producer, expecting both CTAs' bytes)
//                         + the TMA bytes of both CTAs
//   empty[s]  (each CTA)  1 arrival: multicast commit from the even CTA
//   tfull[a]  (each CTA)  1 arrival: multicast commit from the even CTA
//   tempty[a] (even CTA)  16 arrivals: every epilogue warp of both CTAs
// ----------------------------------------------------------------------------
constexpr int BM2 = 256;                 // rows per CTA pair

template <int BN, int EPW, int KSUB>
struct Cfg2 {
    // A stage holds KSUB 64-deep k-blocks (KSUB x 4 MMAs per barrier wait and
    // commit).  8 epilogue warps: 6 stages of one k-block or 3 of two; 16
    // (for the GELU epilogue, which needs more warps to hide its latency): 5
    // or 2, so the epilogue staging fits.
    static constexpr int STAGES = KSUB == 1 ? (EPW == 16 ? 5 : 6) : (EPW == 16 ? 2 : 3);
    static constexpr int THREADS = 128 + 32 * EPW;
    static constexpr int A_SUB = 128 * BK * 2;           // one 64-deep k-block of A (this CTA's 128 rows)
    static constexpr int B_SUB = (BN / 2) * BK * 2;      // ... and of this CTA's half of B
    static constexpr int A_BYTES = KSUB * A_SUB;
    static constexpr int B_BYTES = KSUB * B_SUB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    static constexpr int EPI_BYTES = EPW * 2 * 2048;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr int COLS_PER_WARP = BN / (EPW / 4);   // EPW / 4 warps share a TMEM lane quadrant
    static_assert(EPW == 8 || EPW == 16, "epilogue warps");
    static_assert(KSUB == 1 || KSUB == 2, "k-blocks per stage");
    static_assert(COLS_PER_WARP % 32 == 0, "whole 32-column chunks per warp");
    static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation must be a power of 2");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "pair MMA N");
    static_assert(2 * STAGES * 8 + 4 * 8 + 8 <= BAR_BYTES, "barrier area");
};

template <int BN, int EPI, int EPW, int KSUB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg2<BN, EPW, KSUB>::THREADS, 1)
pffn_gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const Args args) {
    using C = Cfg2<BN, EPW, KSUB>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sA = base;
    const uint32_t sB = base + C::STAGES * C::A_BYTES;
    const uint32_t sEpi = base + C::STAGES * C::STAGE_BYTES;           // epilogue staging, 1024-aligned
    const uint32_t bar0 = sEpi + C::EPI_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES + 8 * (2 * C::STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();          // 0: issues the pair MMAs
    const long long pair = blockIdx.x >> 1;
    const long long npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EPW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();               // reconverge before the aligned cluster barrier
    cluster_sync_all();            // barriers and TMEM of both CTAs exist before any cross-CTA use
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
    pdl_wait();              // operands and outputs are shared with the previous kernels of the stream
    pdl_launch_next();

    const int kblocks = args.K / (BK * KSUB);
    const long long tiles =
        args.tile_prefix ? (long long)__ldg(args.tile_prefix + args.ngroups) * args.n_tiles : args.tiles;

    if (warp == 0) {
        // ---------------------------- TMA producer (both CTAs) ----------------------------
        {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (long long tile = pair; ok && tile < tiles; tile += npairs) {
                const TileCoord tc = decode_tile(tile, args);
                const int arow = args.tile_prefix ? (int)(tc.row0 + (long long)tc.mb * BM2 + 128 * (int)rank)
                                                  : tc.mb * BM2 + 128 * (int)rank;
                const int agrp = args.tile_prefix ? 0 : tc.j;
                const int brow = tc.nb * BN + (BN / 2) * (int)rank;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, args.err, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t fb = mapa_shared(full_bar(stage), 0);
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(2 * C::STAGE_BYTES));
#pragma unroll
                        for (int ks = 0; ks < KSUB; ++ks) {
                            const int kx = (kb * KSUB + ks) * BK;
                            tma_load_3d_pair(&tmA, sA + stage * C::A_BYTES + ks * C::A_SUB, fb, kx, arow, agrp);
                            tma_load_3d_pair(&tmB, sB + stage * C::B_BYTES + ks * C::B_SUB, fb, kx, brow, tc.wg);
                        }
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------- pair MMA issuer (even CTA) --------------------------
        if (rank == 0) {
            constexpr uint32_t idesc = make_idesc_f16_f32(BM2, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (long long tile = pair; ok && tile < tiles; tile += npairs) {
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
                    const uint32_t a0 = sA + stage * C::A_BYTES;
                    const uint32_t b0 = sB + stage * C::B_BYTES;
                    if (lane == 0) {
#pragma unroll
                        for (int ks = 0; ks < KSUB; ++ks)
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k)
                                umma_f16_pair(d_tmem, make_sw128_desc(a0 + ks * C::A_SUB + 32u * k),
                                              make_sw128_desc(b0 + ks * C::B_SUB + 32u * k), idesc,
                                              (kb > 0 || ks > 0 || k > 0) ? 1u : 0u);
                        umma_commit_pair_mc(empty_bar(stage), (uint16_t)0x3);
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) umma_commit_pair_mc(tfull_bar(acc), (uint16_t)0x3);
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else if (warp >= 4) {
        // ---------------------------- epilogue (both CTAs) --------------------------------
        const int ew = warp - 4;
        const int quad = warp & 3;
        const int half = ew >> 2;               // which COLS_PER_WARP columns of the tile
        const int row_in_tile = quad * 32 + lane;
        const uint32_t stage = sEpi + (uint32_t)ew * 4096u;
        int sbuf = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (long long tile = pair; tile < tiles; tile += npairs) {
            const TileCoord tc = decode_tile(tile, args);
            // every lane waits (the warp stays converged for tcgen05.ld)
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.err, args.timeout_ns)) break;
            tc_fence_after();
            const int m = tc.mb * BM2 + 128 * (int)rank + row_in_tile;
            const bool valid = m < tc.Mg;
            const long long arow = tc.row0 + m;
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN + half * C::COLS_PER_WARP);
            const int n0 = tc.nb * BN + half * C::COLS_PER_WARP;
            if (EPI == EPI_GELU && args.hid_tma)
                epilogue_gelu_tma<C::COLS_PER_WARP, EPW == 8>(args, tc, &tmC, tbase, n0, m - lane, stage, lane,
                                                               sbuf);
            else
                epilogue_tile<C::COLS_PER_WARP, EPI>(args, tc, valid, arow, tbase, n0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_group<0>();   // this warp's tensor stores have landed
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();            // no CTA leaves while its peer may still touch its memory
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
// Both FFN GEMMs of a dense layer in one launch (CTA pairs, 256 x 256 tiles,
// 8 epilogue warps): the tile list is every GEMM1 tile (token-major) followed
// by every GEMM2 tile, taken in a static order as in the kernel above.  A
// GEMM2 tile (token j, row block mb) reads the hidden rows that the GEMM1
// tiles (j, mb, every column block) wrote, so:
//   - each epilogue warp of a GEMM1 tile, once its tensor stores of the tile
//     are complete, adds 1 to the row block's counter dep[j m_tiles + mb]
//     (async-proxy fence, then a device-scope fence, then the atomic);
//   - the producer of a GEMM2 tile waits (bounded) until that counter has
//     grown by n_tiles1 x 2 x 8 in this launch, then loads through TMA after
//     an async-proxy fence.
// A warp defers the signal of a GEMM1 tile to its next GEMM1 tile (by then
// the stores have long landed) unless its next tile is not a GEMM1 tile.
// Every GEMM1 tile depends on nothing, and every CTA is resident (one CTA per
// SM, grid <= the SM count), so every wait ends; the bound turns a broken
// assumption into an error instead of a hang.  Counters only grow: launch e
// waits for base + target with base = e x target (wrap-safe comparison); the
// counters of row blocks past this launch's batch get their target too (one
// thread, at the end), so every counter grows by the same amount per launch
// whatever the batch.
// The per-tile arithmetic is that of the two separate launches, so the
// results are the same bits.
// ----------------------------------------------------------------------------
struct LayerDep {
    unsigned* cnt;        // [groups][m_cap]
    unsigned base;        // counter value of a row block at the start of this launch
    unsigned target;      // GEMM1 signals per row block and launch
    int m_cap;            // row blocks per group the counters cover (the context's capacity)
};

__device__ __forceinline__ bool wait_counter_bounded(const unsigned* p, unsigned want, volatile int* abort, int* err,
                                                     uint64_t timeout_ns) {
    if ((int)(ld_acquire_gpu(p) - want) >= 0) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(128);
        if ((int)(ld_acquire_gpu(p) - want) >= 0) return true;
        if ((it & 31u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort = 1;
                latch_error(err, kDevErrTimeout);
                return false;
            }
        }
    }
}

template <int KSUB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg2<256, 8, KSUB>::THREADS, 1)
pffn_layer_tc2_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                      const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ CUtensorMap tmA2,
                      const __grid_constant__ CUtensorMap tmB2, const Args a1, const Args a2, const LayerDep dep) {
    constexpr int BN = 256, EPW = 8;
    using C = Cfg2<BN, EPW, KSUB>;
    constexpr int kGroupsPerTile = C::COLS_PER_WARP / 32;     // tensor-store groups a warp commits per GEMM1 tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sA = base;
    const uint32_t sB = base + C::STAGES * C::A_BYTES;
    const uint32_t sEpi = base + C::STAGES * C::STAGE_BYTES;
    const uint32_t bar0 = sEpi + C::EPI_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES + 8 * (2 * C::STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const long long pair = blockIdx.x >> 1;
    const long long npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmB1);
        tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB2);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EPW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
    pdl_wait();              // S comes from the previous kernel of the stream
    pdl_launch_next();

    const long long tiles1 = a1.tiles, tiles = a1.tiles + a2.tiles;
    const int kblocks1 = a1.K / (BK * KSUB), kblocks2 = a2.K / (BK * KSUB);

    if (warp == 0) {
        // ---------------------------- TMA producer (both CTAs) ----------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long tile = pair; ok && tile < tiles; tile += npairs) {
            const bool g1 = tile < tiles1;
            const Args& a = g1 ? a1 : a2;
            const TileCoord tc = decode_tile(g1 ? tile : tile - tiles1, a);
            const CUtensorMap* mA = g1 ? &tmA1 : &tmA2;
            const CUtensorMap* mB = g1 ? &tmB1 : &tmB2;
            if (!g1) {
                // the hidden rows of (j, mb): every GEMM1 tile of the row block has signalled
                int done = 1;
                if (lane == 0) {
                    done = wait_counter_bounded(dep.cnt + (size_t)tc.j * dep.m_cap + tc.mb, dep.base + dep.target,
                                                abort_flag, a.err, a.timeout_ns) ? 1 : 0;
                    fence_proxy_async_global();
                }
                done = __shfl_sync(0xffffffffu, done, 0);
                if (!done) break;
            }
            const int arow = tc.mb * BM2 + 128 * (int)rank;
            const int brow = tc.nb * BN + (BN / 2) * (int)rank;
            const int kblocks = g1 ? kblocks1 : kblocks2;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.err, a.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(2 * C::STAGE_BYTES));
#pragma unroll
                    for (int ks = 0; ks < KSUB; ++ks) {
                        const int kx = (kb * KSUB + ks) * BK;
                        tma_load_3d_pair(mA, sA + stage * C::A_BYTES + ks * C::A_SUB, fb, kx, arow, tc.j);
                        tma_load_3d_pair(mB, sB + stage * C::B_BYTES + ks * C::B_SUB, fb, kx, brow, tc.wg);
                    }
                }
                __syncwarp();
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------- pair MMA issuer (even CTA) --------------------------
        if (rank == 0) {
            constexpr uint32_t idesc = make_idesc_f16_f32(BM2, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (long long tile = pair; ok && tile < tiles; tile += npairs) {
                const int kblocks = tile < tiles1 ? kblocks1 : kblocks2;
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a1.err, a1.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, a1.err, a1.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * C::A_BYTES;
                    const uint32_t b0 = sB + stage * C::B_BYTES;
                    if (lane == 0) {
#pragma unroll
                        for (int ks = 0; ks < KSUB; ++ks)
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k)
                                umma_f16_pair(d_tmem, make_sw128_desc(a0 + ks * C::A_SUB + 32u * k),
                                              make_sw128_desc(b0 + ks * C::B_SUB + 32u * k), idesc,
                                              (kb > 0 || ks > 0 || k > 0) ? 1u : 0u);
                        umma_commit_pair_mc(empty_bar(stage), (uint16_t)0x3);
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) umma_commit_pair_mc(tfull_bar(acc), (uint16_t)0x3);
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else if (warp >= 4) {
        // ---------------------------- epilogue (both CTAs) --------------------------------
        const int ew = warp - 4;
        const int quad = warp & 3;
        const int half = ew >> 2;
        const int row_in_tile = quad * 32 + lane;
        const uint32_t stage = sEpi + (uint32_t)ew * 4096u;
        int sbuf = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        long long pending = -1;                 // counter of this warp's last GEMM1 tile, not yet signalled
        auto signal = [&](long long idx) {      // lane 0: the stores are complete before this call
            fence_proxy_async_global();
            __threadfence();
            atomicAdd(dep.cnt + idx, 1u);
        };
        for (long long tile = pair; tile < tiles; tile += npairs) {
            const bool g1 = tile < tiles1;
            const Args& a = g1 ? a1 : a2;
            const TileCoord tc = decode_tile(g1 ? tile : tile - tiles1, a);
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, a.err, a.timeout_ns)) break;
            tc_fence_after();
            const int m = tc.mb * BM2 + 128 * (int)rank + row_in_tile;
            const bool valid = m < tc.Mg;
            const long long arow = tc.row0 + m;
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN + half * C::COLS_PER_WARP);
            const int n0 = tc.nb * BN + half * C::COLS_PER_WARP;
            if (g1)
                epilogue_gelu_tma<C::COLS_PER_WARP, true>(a1, tc, &tmC1, tbase, n0, m - lane, stage, lane, sbuf);
            else
                epilogue_tile<C::COLS_PER_WARP, EPI_RESID>(a2, tc, valid, arow, tbase, n0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
            if (g1) {
                if (pending >= 0) {          // the previous GEMM1 tile: all but this tile's groups are complete
                    if (lane == 0) {
                        bulk_wait_group<kGroupsPerTile>();
                        signal(pending);
                    }
                    __syncwarp();
                }
                pending = (long long)tc.j * dep.m_cap + tc.mb;
                if (tile + npairs >= tiles1) {   // the next tile of this pair may wait on this one: signal now
                    if (lane == 0) {
                        bulk_wait_group<0>();
                        signal(pending);
                    }
                    __syncwarp();
                    pending = -1;
                }
            }
        }
        if (lane == 0) {
            bulk_wait_group<0>();   // this warp's tensor stores have landed
            if (pending >= 0) signal(pending);
        }
    } else if (warp == 3 && blockIdx.x == 0 && lane == 0) {
        // the row blocks past this batch: no tile signals them, so they get their target here
        for (int j = 0; j < a1.ngroups; ++j)
            for (int mb = a1.m_tiles; mb < dep.m_cap; ++mb) atomicAdd(dep.cnt + (size_t)j * dep.m_cap + mb, dep.target);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
std::mutex g_mu;
std::string g_err;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        g_err = "cuTensorMapEncodeTiled entry point not available";
        return false;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

// 3-D fp16 tensor map over a [groups][rows][K] buffer (row pitch K elements,
// group pitch group_rows * K), box = 64 (K) x box_rows x 1, 128-byte swizzle.
// Rows past `rows` read as zeros.
bool make_map(CUtensorMap* m, const void* ptr, int K, long long rows, int groups, long long group_rows,
              int box_rows) {
    if (!get_encoder()) return false;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)groups};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)group_rows * (cuuint64_t)K * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lk(g_mu);
        g_err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
        return false;
    }
    return true;
}

// Output map for the hidden activations of uniform groups: fp16 [groups][rows][N]
// (row pitch N, group pitch group_rows * N), box 32 x 32 x 1, 64-byte swizzle.
// Rows at or past `rows` are clipped, so a tile never writes into the next group.
bool make_map_out(CUtensorMap* m, const void* ptr, int N, int rows, int groups, long long group_rows) {
    if (!get_encoder()) return false;
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)rows, (cuuint64_t)groups};
    cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)group_rows * (cuuint64_t)N * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lk(g_mu);
        g_err = "cuTensorMapEncodeTiled (output) failed with CUresult " + std::to_string((int)r);
        return false;
    }
    return true;
}

int pick_bn(int N) {
    if (N % 256 == 0) return 256;
    if (N % 128 == 0) return 128;
    if (N % 64 == 0) return 64;
    return 0;
}

// A: rows_total x K activation rows (row r of launch group j at row0(j) + r);
// W: n_wgroups x N x K weights.
template <int BN, int EPI>
cudaError_t run(const void* A, long long a_rows_total, const void* W, int n_wgroups, Args a, int num_sms,
                cudaStream_t s) {
    using C = Cfg<BN>;
    a.n_tiles = a.N / BN;
    if (a.tile_prefix == nullptr) {
        a.m_tiles = (a.M + BM - 1) / BM;
        a.tiles = (long long)a.ngroups * a.m_tiles * a.n_tiles;
        // Keep the larger operand of a group resident across neighbouring CTAs:
        // walk N fastest when the activation rows (M x K) outweigh the weights (N x K).
        a.n_fastest = a.M > a.N ? 1 : 0;
        if (a.tiles == 0) return cudaSuccess;
    }
    CUtensorMap mA, mB, mC;
    const bool a_uniform = a.tile_prefix == nullptr;
    if (!make_map(&mA, A, a.K, a_uniform ? a.M : a_rows_total, a_uniform ? a.ngroups : 1,
                  a_uniform ? a.a_group_rows : a_rows_total, BM))
        return cudaErrorInvalidValue;
    if (!make_map(&mB, W, a.K, a.N, n_wgroups, a.N, BN)) return cudaErrorInvalidValue;
    if (EPI == EPI_GELU && a.hid_tma && a.tile_prefix == nullptr) {
        if (!make_map_out(&mC, a.hid, a.N, a.M, a.ngroups, a.a_group_rows)) return cudaErrorInvalidValue;
    } else {
        a.hid_tma = 0;
        mC = mA;   // unused
    }
    auto k = pffn_gemm_tc_kernel<BN, EPI>;
    {
        cudaError_t e = smem_attr_once((const void*)k, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    long long grid = num_sms;
    if (a.tile_prefix == nullptr && a.tiles < grid) grid = a.tiles;
    return launch_k(k, dim3((unsigned)grid), dim3(kThreads), C::SMEM_BYTES, s, mA, mB, mC, a);
}

template <int EPI>
cudaError_t run_bn(int bn, const void* A, long long a_rows_total, const void* W, int n_wgroups, const Args& a,
                   int num_sms, cudaStream_t s) {
    switch (bn) {
        case 256: return run<256, EPI>(A, a_rows_total, W, n_wgroups, a, num_sms, s);
        case 128: return run<128, EPI>(A, a_rows_total, W, n_wgroups, a, num_sms, s);
        case 64: return run<64, EPI>(A, a_rows_total, W, n_wgroups, a, num_sms, s);
        default: return cudaErrorNotSupported;
    }
}


// CTA-pair launch for uniform groups (dense PFFN).  Grid = 2 x the number of
// pairs that can be resident at once (persistent).
template <int BN, int EPI, int EPW, int KSUB>
cudaError_t run_pair(const void* A, long long a_rows_total, const void* W, int n_wgroups, Args a, int num_sms,
                     cudaStream_t s) {
    using C = Cfg2<BN, EPW, KSUB>;
    if (a.K % (BK * KSUB) != 0) return cudaErrorInvalidValue;
    a.n_tiles = a.N / BN;
    if (a.tile_prefix == nullptr) {        // uniform groups
        a.m_tiles = (a.M + BM2 - 1) / BM2;
        a.tiles = (long long)a.ngroups * a.m_tiles * a.n_tiles;
        a.n_fastest = a.M > a.N ? 1 : 0;
        if (a.tiles == 0) return cudaSuccess;
    } else {                               // variable groups: a.tile_prefix counts 256-row tiles,
        a.tiles = 0;                       // the kernel reads the total; persistent grid
        a.hid_tma = 0;
    }
    CUtensorMap mA, mB, mC;
    const bool a_uniform = a.tile_prefix == nullptr;
    if (!make_map(&mA, A, a.K, a_uniform ? a.M : a_rows_total, a_uniform ? a.ngroups : 1,
                  a_uniform ? a.a_group_rows : a_rows_total, 128))
        return cudaErrorInvalidValue;
    if (!make_map(&mB, W, a.K, a.N, n_wgroups, a.N, BN / 2)) return cudaErrorInvalidValue;
    if (EPI == EPI_GELU && a.hid_tma) {
        if (!make_map_out(&mC, a.hid, a.N, a.M, a.ngroups, a.a_group_rows)) return cudaErrorInvalidValue;
    } else {
        a.hid_tma = 0;
        mC = mA;   // unused
    }
    auto k = pffn_gemm_tc2_kernel<BN, EPI, EPW, KSUB>;
    {
        cudaError_t e = smem_attr_once((const void*)k, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    const int max_pairs = pair_occupancy_once((const void*)k, C::THREADS, C::SMEM_BYTES, num_sms);
    long long pairs = (a.tile_prefix == nullptr && a.tiles < max_pairs) ? a.tiles : max_pairs;
    return launch_k(k, dim3((unsigned)(2 * pairs)), dim3(C::THREADS), C::SMEM_BYTES, s, mA, mB, mC, a);
}

// Pair tiles (256 x BN per CTA pair) for both GEMMs when every token group
// has at least 256 rows.  RM_GEMM_PAIR in the environment overrides the
// choice: 0 never, 2 the second GEMM only (a tuning and diagnosis switch;
// every choice computes the same result).
bool use_pair(int M, int epi) {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_GEMM_PAIR");
        env = !v ? 1 : (v[0] == '0' ? 0 : (v[0] == '2' ? 2 : 1));
    }
    if (M < BM2 || env == 0) return false;
    return env == 1 || epi == EPI_RESID;
}

// The GELU pair kernel's epilogue (a 128 x BN tile per CTA through 8 warps)
// takes about as long as the MMAs of a 256 x 256 x 768 tile: with K = D <=
// kShortK the tile's k-loop is too short to hide it, so that GEMM runs 16
// epilogue warps and, to fit their staging, 5 stages of one k-block each.
// Measured on GB300 at the 100M shape (T=16, D=768, B=2048): GEMM1 4-5% faster
// than with 8 warps and 3 two-k-block stages; at D = 1536 the 8-warp form is
// 16% faster.
constexpr int kShortK = 1024;

// Two 64-deep k-blocks per pipeline stage (when K allows): half the barrier
// waits and commits per MMA, 3 stages of 64 KB per CTA.  Measured on GB300
// (ncu, B = 2048 at the 1B shape, tensor pipe busy): the first GEMM 91.8%
// against 80.2% with 6 stages of one k-block (74.2% with one CTA per tile),
// the second 88.6% against 86.8%.  RM_GEMM_KSUB=1|2 in the environment forces
// one or two k-blocks per stage (a tuning switch; the same result either way).
bool use_ksub2(int K, int epi) {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_GEMM_KSUB");
        env = !v ? 0 : (v[0] == '1' ? 1 : (v[0] == '2' ? 2 : 0));
    }
    if (K % (2 * BK) != 0) return false;
    if (env != 0) return env == 2;
    return !(epi == EPI_GELU && K <= kShortK);
}

// Epilogue warps of the GELU pair kernel: 16 when K <= kShortK, else 8;
// RM_GEMM1_EPW=8|16 in the environment forces either (a tuning switch; the
// same result either way).
bool gelu_pair_epw16(int K) {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_GEMM1_EPW");
        env = !v ? 0 : ((v[0] == '1' && v[1] == '6') ? 16 : (v[0] == '8' ? 8 : 0));
    }
    if (env != 0) return env == 16;
    return K <= kShortK;
}

template <int EPI, int EPW>
cudaError_t run_pair_bn(int bn, bool k2, const void* A, long long a_rows_total, const void* W, int n_wgroups,
                        const Args& a, int num_sms, cudaStream_t s) {
    switch (bn) {
        case 256:
            return k2 ? run_pair<256, EPI, EPW, 2>(A, a_rows_total, W, n_wgroups, a, num_sms, s)
                      : run_pair<256, EPI, EPW, 1>(A, a_rows_total, W, n_wgroups, a, num_sms, s);
        case 128:
            return k2 ? run_pair<128, EPI, EPW, 2>(A, a_rows_total, W, n_wgroups, a, num_sms, s)
                      : run_pair<128, EPI, EPW, 1>(A, a_rows_total, W, n_wgroups, a, num_sms, s);
        case 64:
            return k2 ? run_pair<64, EPI, 8, 2>(A, a_rows_total, W, n_wgroups, a, num_sms, s)
                      : run_pair<64, EPI, 8, 1>(A, a_rows_total, W, n_wgroups, a, num_sms, s);
        default: return cudaErrorNotSupported;
    }
}

// ----------------------------------------------------------------------------
// Small batches: the weights as the MMA's M side.  With B rows per token group
// the 128-row activation tile of the kernels above is mostly zeros: the time
// goes into streaming the weights, and the A tile's shared-memory slots (16 KB
// a stage, loaded as zero fill) crowd out weight stages.  Here D^T = W^T S^T:
// a work unit is 128 output features of one token group; the MMA takes 128
// weight rows (A, K-major, as packed) against NB activation rows (B, K-major,
// NB = B rounded up to a legal N), accumulates 128 x NB in TMEM, and a stage
// is 16 KB of weights + NB x 128 B of activations, so 8-11 stages of weights
// are in flight per SM.  Units walk the feature blocks of a token group
// fastest (its activation rows stay in L2).
//   warp 0      TMA producer
//   warp 1      MMA issuer (one thread)
//   warp 2      TMEM allocator
//   warps 4..   epilogue, 4 warps (8 for NB >= 64, two per TMEM lane quadrant
//               splitting the columns): warp 4 + e reads TMEM lanes 32 q .. 32 q
//               + 31 (q = e mod 4, one feature per lane) and its share of the NB
//               batch columns; GEMM1 stores
//               Gelu(acc + b1) per (row, feature), GEMM2 stores acc + b2 + S and
//               the (mean, M2) of each row over the unit's 128 features (the
//               128-column statistics chunk of the two-phase LN2), the four
//               warps' partial moments merged by Chan's formula in shared memory.
// ----------------------------------------------------------------------------
template <int NB>
struct CfgS {
    static constexpr int A_BYTES = 128 * BK * 2;
    static constexpr int B_BYTES = NB * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int STAT_BYTES = 2 * 2 * 4 * NB * 4;     // (mean, M2) x 2 buffers x 4 warps x NB
    // as many stages (weight bytes in flight) as shared memory takes, at most 12
    static constexpr int STAGE_ROOM = (227 * 1024 - 1024 - BAR_BYTES - STAT_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGE_ROOM > 12 ? 12 : STAGE_ROOM;
    static constexpr int TMEM_COLS = 2 * NB < 32 ? 32 : 2 * NB;
    static constexpr int EPW = NB >= 64 ? 8 : 4;             // epilogue warps
    static constexpr int CPW = NB / (EPW / 4);               // batch columns per epilogue warp
    static constexpr int THREADS = 128 + 32 * EPW;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + STAT_BYTES;
    static_assert(NB % 16 == 0 && NB >= 16 && NB <= 256, "MMA N for M = 128");
    static_assert(B_BYTES % 1024 == 0, "swizzle atoms of the activation tile");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM allocation");
    static_assert(2 * STAGES * 8 + 4 * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// 16 consecutive fp32 TMEM columns of this thread's lane (32x32b shape, x16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One work unit's epilogue for one epilogue warp of the weights-as-M kernels:
// TMEM lanes 32 q .. 32 q + 31 (feature f = 128 fb + 32 q + lane of this lane)
// and the warp's batch columns col0 .. col0 + CPW - 1 of the accumulator at
// tbase; s_stat_acc is the accumulator buffer's slice of the row-moment area.
template <int NB, int EPI>
__device__ __forceinline__ void swap_epilogue_unit(const Args& args, int fb, int f, float bf, size_t row0, bool uok,
                                                   uint32_t tbase, float* s_stat_acc, int q, int col0, int lane) {
    using C = CfgS<NB>;
    constexpr int CW = NB < 32 ? NB : 32;        // TMEM columns per load
    float* st_mean = s_stat_acc + (size_t)q * NB;
    float* st_m2 = st_mean + 4 * NB;
#pragma unroll 1
    for (int c = col0; c < col0 + C::CPW && c < args.M; c += CW) {
        float v[CW];
        if constexpr (CW == 32) {
            tmem_ld32(tbase + (uint32_t)c, v);
        } else {
            tmem_ld16(tbase + (uint32_t)c, v);
        }
        if (EPI == EPI_GELU) {
            // two batch rows at a time through the packed GELU
#pragma unroll
            for (int i = 0; i < CW; i += 2) {
                const int b = c + i;                               // batch row (warp-uniform)
                if (b >= args.M) break;
                float g0, g1;
                f2_unpack(gelu_erf_x2(f2_pack(v[i], v[i + 1]), f2_splat(bf)), g0, g1);
                if (uok) args.hid[(row0 + b) * (size_t)args.N + f] = __float2half_rn(sat_f16(g0));
                if (uok && b + 1 < args.M)
                    args.hid[(row0 + b + 1) * (size_t)args.N + f] = __float2half_rn(sat_f16(g1));
            }
        } else {   // EPI_RESID
            // the residuals of the chunk's rows first, all loads in flight together
            float rres[CW];
#pragma unroll
            for (int i = 0; i < CW; ++i) {
                const int b = c + i;
                rres[i] = (uok && b < args.M) ? __half2float(args.resid[(row0 + b) * (size_t)args.N + f]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < CW; ++i) {
                const int b = c + i;                               // batch row (warp-uniform)
                if (b >= args.M) break;
                const float z = v[i] + bf + rres[i];
                if (uok) args.z[(row0 + b) * (size_t)args.N + f] = __float2half_rn(sat_f16(z));
                // this warp's 32 features: mean and M2 about it
                const float mw = warp_sum(z) * (1.0f / 32.0f);
                const float d = z - mw;
                const float m2w = warp_sum(d * d);
                if (lane == 0) {
                    st_mean[b] = mw;
                    st_m2[b] = m2w;
                }
            }
        }
    }
    if (EPI == EPI_RESID) {
        // the four quadrants' moments -> (mean, M2) of the 128 features, one lane
        // per row, each q = 0 warp for its own columns
        asm volatile("bar.sync 1, %0;" ::"r"(C::EPW * 32) : "memory");
        if (q == 0) {
            const float* sm = s_stat_acc;
            const float* s2 = sm + 4 * NB;
            for (int b = col0 + lane; b < args.M && b < col0 + C::CPW; b += 32) {
                const float m0 = sm[b], m1 = sm[NB + b], m2 = sm[2 * NB + b], m3 = sm[3 * NB + b];
                const float mean = 0.25f * (m0 + m1 + m2 + m3);
                const float d0 = m0 - mean, d1 = m1 - mean, d2 = m2 - mean, d3 = m3 - mean;
                const float M2 = s2[b] + s2[NB + b] + s2[2 * NB + b] + s2[3 * NB + b] +
                                 32.0f * (d0 * d0 + d1 * d1 + d2 * d2 + d3 * d3);
                if (uok) args.stats[(row0 + b) * (size_t)args.nchunk + fb] = make_float2(mean, M2);
            }
        }
    }
}

template <int NB, int EPI>
__global__ void __launch_bounds__(CfgS<NB>::THREADS, 1)
pffn_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const Args args) {
    using C = CfgS<NB>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sA = base;
    const uint32_t sB = base + C::STAGES * C::A_BYTES;
    const uint32_t bar0 = base + C::STAGES * C::STAGE_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::STAGES * C::STAGE_BYTES + 8 * (2 * C::STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // per-warp row moments of the last GEMM's units: [buffer][mean | M2][warp][NB]
    float* s_stat = reinterpret_cast<float*>(base_ptr + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), C::EPW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
    pdl_wait();              // operands and outputs are shared with the previous kernels of the stream
    pdl_launch_next();

    const int kblocks = args.K / BK;
    const long long units = args.tiles;             // token groups x feature blocks
    const int nfb = args.n_tiles;                   // feature blocks of 128 per group

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int j = (int)(u / nfb);
            const int fb = (int)(u - (long long)j * nfb);
            const int wg = args.group_base + j * args.group_stride;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, args.err, args.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage), (uint32_t)C::STAGE_BYTES);
                    tma_load_3d(&tmW, sA + stage * C::A_BYTES, full_bar(stage), kb * BK, fb * 128, wg);
                    tma_load_3d(&tmX, sB + stage * C::B_BYTES, full_bar(stage), kb * BK, 0, j);
                }
                __syncwarp();
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        constexpr uint32_t idesc = make_idesc_f16_f32(128, NB);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (long long u = blockIdx.x; ok && u < units; u += gridDim.x) {
            if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err, args.timeout_ns)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NB);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.err, args.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sA + stage * C::A_BYTES;
                const uint32_t b0 = sB + stage * C::B_BYTES;
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_f16(d_tmem, make_sw128_desc(a0 + 32u * k), make_sw128_desc(b0 + 32u * k), idesc,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (lane == 0) umma_commit(tfull_bar(acc));
            __syncwarp();
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    } else if (warp >= 4) {
        // ------------------------------ epilogue ----------------------------------
        const int e = warp - 4;
        const int q = warp & 3;                       // TMEM lane quadrant
        const int col0 = (e >> 2) * C::CPW;           // this warp's first batch column
        int acc = 0;
        uint32_t acc_phase = 0;
        for (long long u = blockIdx.x; u < units; u += gridDim.x) {
            const int j = (int)(u / nfb);
            const int fb = (int)(u - (long long)j * nfb);
            const int wg = args.group_base + j * args.group_stride;
            const int f = fb * 128 + q * 32 + lane;                      // this lane's output feature
            const float bf = __ldg(args.bias + (size_t)wg * args.N + f);
            const size_t row0 = (size_t)j * (size_t)args.a_group_rows;   // row of batch 0 of this group
            // bounds-checked build: the unit's rows and features lie inside the buffers
            const bool uok = RM_IN_BOUNDS((long long)row0 + args.M <= args.rows_cap && args.M <= args.a_group_rows &&
                                              fb * 128 + 128 <= args.N, args.err);
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.err, args.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * NB);
            swap_epilogue_unit<NB, EPI>(args, fb, f, bf, row0, uok, tbase, s_stat + (size_t)acc * 2 * 4 * NB, q, col0,
                                        lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
// Both FFN GEMMs of a dense layer in one launch for small batches (weights as
// M, the units of the kernel above): the unit list is every GEMM1 unit (token
// j, 128 hidden features; token-major) followed by every GEMM2 unit (token j,
// 128 output features), taken in a static order, so the second GEMM's units
// fill the SMs that the first leaves idle instead of starting a launch of
// their own with 2.5 rounds of units.  A GEMM2 unit of token j reads the
// hidden rows of every GEMM1 unit of token j:
//   - each epilogue warp of a GEMM1 unit, after its stores of the unit, makes
//     them visible device-wide (every lane fences) and adds 8 / EPW to the
//     token's counter dep[j m_cap], so a unit adds 8 and a token F / 16 --
//     the target per row block of the CTA-pair layer kernel, whose counters
//     and epochs these are (row block 0; the others get their target from
//     one thread);
//   - the producer of a GEMM2 unit waits (bounded) until the counter has
//     grown by the target in this launch, then loads through TMA after an
//     async-proxy fence.
// GEMM1 units wait on nothing and every CTA is resident (one per SM, grid <=
// the SM count), so every wait ends.  Per unit the arithmetic is that of the
// two separate launches: the same bits.
// ----------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(CfgS<NB>::THREADS, 1)
pffn_layer_swap_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmX1,
                       const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmX2,
                       const Args a1, const Args a2, const LayerDep dep) {
    using C = CfgS<NB>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sA = base;
    const uint32_t sB = base + C::STAGES * C::A_BYTES;
    const uint32_t bar0 = base + C::STAGES * C::STAGE_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::STAGES * C::STAGE_BYTES + 8 * (2 * C::STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* s_stat = reinterpret_cast<float*>(base_ptr + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW1);
        tma_prefetch_desc(&tmX1);
        tma_prefetch_desc(&tmW2);
        tma_prefetch_desc(&tmX2);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), C::EPW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
    pdl_wait();              // S comes from the previous kernel of the stream
    pdl_launch_next();

    const int nfb1 = a1.n_tiles, nfb2 = a2.n_tiles;        // feature blocks of 128 per token
    const long long units1 = a1.tiles, units = a1.tiles + a2.tiles;
    const int kblocks1 = a1.K / BK, kblocks2 = a2.K / BK;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const bool g1 = u < units1;
            const Args& a = g1 ? a1 : a2;
            const long long uu = g1 ? u : u - units1;
            const int nfb = g1 ? nfb1 : nfb2;
            const int j = (int)(uu / nfb);
            const int fb = (int)(uu - (long long)j * nfb);
            const int wg = a.group_base + j * a.group_stride;
            if (!g1) {
                // the hidden rows of token j: every GEMM1 unit of the token has signalled
                int done = 1;
                if (lane == 0) {
                    done = wait_counter_bounded(dep.cnt + (size_t)j * dep.m_cap, dep.base + dep.target, abort_flag,
                                                a.err, a.timeout_ns) ? 1 : 0;
                    fence_proxy_async_global();
                }
                done = __shfl_sync(0xffffffffu, done, 0);
                if (!done) break;
            }
            const CUtensorMap* mW = g1 ? &tmW1 : &tmW2;
            const CUtensorMap* mX = g1 ? &tmX1 : &tmX2;
            const int kblocks = g1 ? kblocks1 : kblocks2;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.err, a.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage), (uint32_t)C::STAGE_BYTES);
                    tma_load_3d(mW, sA + stage * C::A_BYTES, full_bar(stage), kb * BK, fb * 128, wg);
                    tma_load_3d(mX, sB + stage * C::B_BYTES, full_bar(stage), kb * BK, 0, j);
                }
                __syncwarp();
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        constexpr uint32_t idesc = make_idesc_f16_f32(128, NB);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (long long u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int kblocks = u < units1 ? kblocks1 : kblocks2;
            if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a1.err, a1.timeout_ns)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NB);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, a1.err, a1.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sA + stage * C::A_BYTES;
                const uint32_t b0 = sB + stage * C::B_BYTES;
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_f16(d_tmem, make_sw128_desc(a0 + 32u * k), make_sw128_desc(b0 + 32u * k), idesc,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (lane == 0) umma_commit(tfull_bar(acc));
            __syncwarp();
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    } else if (warp >= 4) {
        // ------------------------------ epilogue ----------------------------------
        const int e = warp - 4;
        const int q = warp & 3;                       // TMEM lane quadrant
        const int col0 = (e >> 2) * C::CPW;           // this warp's first batch column
        constexpr unsigned kSignal = 8u / (unsigned)C::EPW;   // per warp: 8 per unit
        static_assert(8 % C::EPW == 0, "signal per unit");
        int acc = 0;
        uint32_t acc_phase = 0;
        for (long long u = blockIdx.x; u < units; u += gridDim.x) {
            const bool g1 = u < units1;
            const Args& a = g1 ? a1 : a2;
            const long long uu = g1 ? u : u - units1;
            const int nfb = g1 ? nfb1 : nfb2;
            const int j = (int)(uu / nfb);
            const int fb = (int)(uu - (long long)j * nfb);
            const int wg = a.group_base + j * a.group_stride;
            const int f = fb * 128 + q * 32 + lane;                      // this lane's output feature
            const float bf = __ldg(a.bias + (size_t)wg * a.N + f);
            const size_t row0 = (size_t)j * (size_t)a.a_group_rows;      // row of batch 0 of this group
            const bool uok = RM_IN_BOUNDS((long long)row0 + a.M <= a.rows_cap && a.M <= a.a_group_rows &&
                                              fb * 128 + 128 <= a.N, a.err);
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, a.err, a.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * NB);
            float* st = s_stat + (size_t)acc * 2 * 4 * NB;
            if (g1)
                swap_epilogue_unit<NB, EPI_GELU>(a1, fb, f, bf, row0, uok, tbase, st, q, col0, lane);
            else
                swap_epilogue_unit<NB, EPI_RESID>(a2, fb, f, bf, row0, uok, tbase, st, q, col0, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
            if (g1) {
                // this warp's hidden rows of the unit are stored: publish them, then count
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(dep.cnt + (size_t)j * dep.m_cap, kSignal);
            }
        }
    } else if (warp == 3 && blockIdx.x == 0 && lane == 0) {
        // row blocks 1 .. m_cap - 1 of every token: no unit signals them, so they get their target here
        for (int j = 0; j < a1.ngroups; ++j)
            for (int mb = 1; mb < dep.m_cap; ++mb) atomicAdd(dep.cnt + (size_t)j * dep.m_cap + mb, dep.target);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Largest batch that takes the weight-as-M path (RM_GEMM_SWAP_MAX in the
// environment overrides; 0 turns it off -- a tuning switch, the same result
// up to the fp32 summation order).
int swap_max_batch() {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_GEMM_SWAP_MAX");
        env = v ? atoi(v) : 64;
        if (env > 256) env = 256;
    }
    return env;
}

template <int NB, int EPI>
cudaError_t run_swap(const void* A, const void* W, int n_wgroups, Args a, int num_sms, cudaStream_t s) {
    using C = CfgS<NB>;
    a.n_tiles = a.N / 128;
    a.tiles = (long long)a.ngroups * a.n_tiles;
    if (a.tiles == 0) return cudaSuccess;
    CUtensorMap mW, mX;
    if (!make_map(&mW, W, a.K, a.N, n_wgroups, a.N, 128)) return cudaErrorInvalidValue;
    if (!make_map(&mX, A, a.K, a.M, a.ngroups, a.a_group_rows, NB)) return cudaErrorInvalidValue;
    auto k = pffn_gemm_swap_kernel<NB, EPI>;
    {
        cudaError_t e = smem_attr_once((const void*)k, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    const long long grid = a.tiles < num_sms ? a.tiles : num_sms;
    return launch_k(k, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, s, mW, mX, a);
}

template <int EPI>
cudaError_t run_swap_nb(const void* A, const void* W, int n_wgroups, const Args& a, int num_sms, cudaStream_t s) {
    if (a.M <= 16) return run_swap<16, EPI>(A, W, n_wgroups, a, num_sms, s);
    if (a.M <= 32) return run_swap<32, EPI>(A, W, n_wgroups, a, num_sms, s);
    if (a.M <= 64) return run_swap<64, EPI>(A, W, n_wgroups, a, num_sms, s);
    if (a.M <= 128) return run_swap<128, EPI>(A, W, n_wgroups, a, num_sms, s);
    return run_swap<256, EPI>(A, W, n_wgroups, a, num_sms, s);
}

template <int EPI>
cudaError_t run_dense(int bn, const void* A, long long a_rows_total, const void* W, int n_wgroups, const Args& a,
                      int num_sms, cudaStream_t s) {
    // weights as the MMA's M side for small batches; the second GEMM's row
    // statistics then come in 128-column chunks, which must be the context's
    if (a.M <= swap_max_batch() && a.N % 128 == 0 && a.K % BK == 0 &&
        (EPI == EPI_GELU || (EPI == EPI_RESID && a.nchunk * 128 == a.N)))
        return run_swap_nb<EPI>(A, W, n_wgroups, a, num_sms, s);
    if (use_pair(a.M, EPI)) {
        const bool k2 = use_ksub2(a.K, EPI);
        if (EPI == EPI_GELU && gelu_pair_epw16(a.K))
            return run_pair_bn<EPI, 16>(bn, k2, A, a_rows_total, W, n_wgroups, a, num_sms, s);
        return run_pair_bn<EPI, 8>(bn, k2, A, a_rows_total, W, n_wgroups, a, num_sms, s);
    }
    // RM_GEMM_SMALL_BN=64|128: narrower one-CTA tiles for the first GEMM (a tuning
    // switch; the second GEMM's tile width fixes its statistics chunks, see gemm2_bn)
    static int small_bn = -1;
    if (small_bn < 0) {
        const char* v = getenv("RM_GEMM_SMALL_BN");
        small_bn = v ? atoi(v) : 0;
    }
    if (EPI == EPI_GELU && (small_bn == 64 || small_bn == 128) && small_bn < bn && a.N % small_bn == 0)
        bn = small_bn;
    return run_bn<EPI>(bn, A, a_rows_total, W, n_wgroups, a, num_sms, s);
}

// Both FFN GEMMs of a layer in one launch (pffn_layer_tc2_kernel) whenever
// both would run as 256 x 256 CTA-pair tiles; RM_GEMM_FUSED=0 in the
// environment keeps the two launches (a tuning switch: the same bits).
bool fused_enabled() {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_GEMM_FUSED");
        env = (v && v[0] == '0') ? 0 : 1;
    }
    return env == 1;
}

template <int KSUB>
cudaError_t run_layer(const void* S, const void* W1p, const void* W2p, Args a1, Args a2, unsigned* dep_cnt,
                      unsigned dep_epoch, int num_sms, cudaStream_t s) {
    using C = Cfg2<256, 8, KSUB>;
    CUtensorMap mA1, mB1, mC1, mA2, mB2;
    if (!make_map(&mA1, S, a1.K, a1.M, a1.ngroups, a1.a_group_rows, 128) ||
        !make_map(&mB1, W1p, a1.K, a1.N, a1.ngroups, a1.N, 128) ||
        !make_map_out(&mC1, a1.hid, a1.N, a1.M, a1.ngroups, a1.a_group_rows) ||
        !make_map(&mA2, a1.hid, a2.K, a2.M, a2.ngroups, a2.a_group_rows, 128) ||
        !make_map(&mB2, W2p, a2.K, a2.N, a2.ngroups, a2.N, 128))
        return cudaErrorInvalidValue;
    LayerDep dep;
    dep.cnt = dep_cnt;
    dep.target = (unsigned)a1.n_tiles * 2u * 8u;
    dep.base = dep_epoch * dep.target;
    dep.m_cap = (int)((a1.a_group_rows + BM2 - 1) / BM2);
    auto k = pffn_layer_tc2_kernel<KSUB>;
    {
        cudaError_t e = smem_attr_once((const void*)k, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    const int max_pairs = pair_occupancy_once((const void*)k, C::THREADS, C::SMEM_BYTES, num_sms);
    const long long tiles = a1.tiles + a2.tiles;
    const long long pairs = tiles < max_pairs ? tiles : max_pairs;
    return launch_k(k, dim3((unsigned)(2 * pairs)), dim3(C::THREADS), C::SMEM_BYTES, s, mA1, mB1, mC1, mA2, mB2, a1,
                    a2, dep);
}

template <int NB>
cudaError_t run_layer_swap(const void* S, const void* W1p, const void* W2p, Args a1, Args a2, unsigned* dep_cnt,
                           unsigned dep_epoch, int num_sms, cudaStream_t s) {
    using C = CfgS<NB>;
    a1.n_tiles = a1.N / 128;
    a1.tiles = (long long)a1.ngroups * a1.n_tiles;
    a2.n_tiles = a2.N / 128;
    a2.tiles = (long long)a2.ngroups * a2.n_tiles;
    CUtensorMap mW1, mX1, mW2, mX2;
    if (!make_map(&mW1, W1p, a1.K, a1.N, a1.ngroups, a1.N, 128) ||
        !make_map(&mX1, S, a1.K, a1.M, a1.ngroups, a1.a_group_rows, NB) ||
        !make_map(&mW2, W2p, a2.K, a2.N, a2.ngroups, a2.N, 128) ||
        !make_map(&mX2, a1.hid, a2.K, a2.M, a2.ngroups, a2.a_group_rows, NB))
        return cudaErrorInvalidValue;
    LayerDep dep;
    dep.cnt = dep_cnt;
    dep.target = (unsigned)a1.n_tiles * 8u;     // = F / 16, the CTA-pair layer kernel's target
    dep.base = dep_epoch * dep.target;
    dep.m_cap = (int)((a1.a_group_rows + BM2 - 1) / BM2);
    auto k = pffn_layer_swap_kernel<NB>;
    {
        cudaError_t e = smem_attr_once((const void*)k, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    const long long units = a1.tiles + a2.tiles;
    const long long grid = units < num_sms ? units : num_sms;   // one CTA per SM: all resident
    return launch_k(k, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, s, mW1, mX1, mW2, mX2, a1, a2, dep);
}

}  // namespace tc

int gemm2_bn(int D);

// The hidden layer's tensor stores carry the L2 evict-first hint when the
// layer's hidden rows (B T F fp16 values) exceed 128 MB, i.e. L2: they are
// read back only after every first-GEMM tile, so L2 could not keep them
// anyway.  RM_HID_HINT=0 | 1 in the environment forces either (a tuning
// switch: the same results).
bool hid_evict_first(int B, int T, int F) {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_HID_HINT");
        env = !v ? 2 : (v[0] == '0' ? 0 : 1);
    }
    if (env != 2) return env == 1;
    return (long long)B * T * F * 2 > (128LL << 20);
}

bool layer_tc_fusable(int B, int D, int F) {
    if (!tc::fused_enabled()) return false;
    // weights as M (128-feature units, 128-column LN2 chunks): fused from B = 17 on.  At the
    // 1B shape, B = 64: 0.451 against 0.466 ms per step; B = 1 and 8: 0.410 / 0.426 against
    // 0.410 / 0.423 (the separate launches overlap more with their neighbours there).
    if (B <= tc::swap_max_batch())
        return B > 16 && D % 128 == 0 && F % 128 == 0 && gemm2_bn(D) == 256 && F % 256 == 0;
    return tc::use_pair(B, tc::EPI_GELU) && tc::use_pair(B, tc::EPI_RESID) && tc::pick_bn(F) == 256 &&
           gemm2_bn(D) == 256 && D % (2 * tc::BK) == 0 && F % (2 * tc::BK) == 0;
}

cudaError_t launch_layer_tc(const void* S, const void* W1p, const float* b1, void* Hid, const void* W2p,
                            const float* b2, void* Z, float2* stats, int B, int T, int D, int F, int Bcap, int num_sms,
                            unsigned* dep_cnt, unsigned dep_epoch, int* err, unsigned long long timeout_ns,
                            cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (!layer_tc_fusable(B, D, F) || !dep_cnt) return cudaErrorNotSupported;
    RM_HOST_BOUNDS(B <= Bcap && S && W1p && b1 && Hid && W2p && b2 && Z && stats);
    RM_HOST_BOUNDS(((reinterpret_cast<uintptr_t>(S) | reinterpret_cast<uintptr_t>(W1p) | reinterpret_cast<uintptr_t>(Hid) |
                     reinterpret_cast<uintptr_t>(W2p) | reinterpret_cast<uintptr_t>(Z)) & 15u) == 0);
    tc::Args a1{}, a2{};
    a1.N = F;
    a1.K = D;
    a1.ngroups = T;
    a1.group_base = 0;
    a1.group_stride = 1;
    a1.M = B;
    a1.a_group_rows = Bcap;
    a1.bias = b1;
    a1.hid = reinterpret_cast<__half*>(Hid);
    a1.hid_tma = 1;
    a1.hid_evict_first = hid_evict_first(B, T, F) ? 1 : 0;
    a1.rows_cap = (long long)T * Bcap;
    a1.err = err;
    a1.timeout_ns = timeout_ns;
    a1.n_tiles = F / 256;
    a1.m_tiles = (B + tc::BM2 - 1) / tc::BM2;
    a1.tiles = (long long)T * a1.m_tiles * a1.n_tiles;
    a1.n_fastest = a1.M > a1.N ? 1 : 0;
    a2.N = D;
    a2.K = F;
    a2.ngroups = T;
    a2.group_base = 0;
    a2.group_stride = 1;
    a2.M = B;
    a2.a_group_rows = Bcap;
    a2.bias = b2;
    a2.resid = reinterpret_cast<const __half*>(S);
    a2.z = reinterpret_cast<__half*>(Z);
    a2.stats = stats;
    a2.nchunk = D / 128;
    a2.rows_cap = (long long)T * Bcap;
    a2.err = err;
    a2.timeout_ns = timeout_ns;
    a2.n_tiles = D / 256;
    a2.m_tiles = a1.m_tiles;
    a2.tiles = (long long)T * a2.m_tiles * a2.n_tiles;
    a2.n_fastest = a2.M > a2.N ? 1 : 0;
    if (B <= tc::swap_max_batch()) {
        if (B <= 16) return tc::run_layer_swap<16>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s);
        if (B <= 32) return tc::run_layer_swap<32>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s);
        if (B <= 64) return tc::run_layer_swap<64>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s);
        if (B <= 128) return tc::run_layer_swap<128>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s);
        return tc::run_layer_swap<256>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s);
    }
    // one stage depth for both GEMMs: two k-blocks a stage unless RM_GEMM_KSUB=1
    const bool k2 = tc::use_ksub2(F, tc::EPI_RESID) && D % (2 * tc::BK) == 0;
    return k2 ? tc::run_layer<2>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s)
              : tc::run_layer<1>(S, W1p, W2p, a1, a2, dep_cnt, dep_epoch, num_sms, s);
}

bool tc_supported(int D, int F) {
    return D % tc::BK == 0 && F % tc::BK == 0 && tc::pick_bn(F) != 0 && tc::pick_bn(D) != 0;
}

// Tile width of the second GEMM (N = D): the widest of 256, 128, 64 dividing D;
// RM_GEMM2_BN=128|64 in the environment narrows it (a tuning switch; the
// statistics chunks follow the tile, so every choice gives the same rows).
int gemm2_bn(int D) {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_GEMM2_BN");
        env = v ? atoi(v) : 0;
    }
    const int bn = tc::pick_bn(D);
    if ((env == 128 || env == 64) && env < bn && D % env == 0) return env;
    return bn;
}

int tc_stats_chunk_width(int D) { return gemm2_bn(D) / 2; }

const char* tc_last_error() {
    std::lock_guard<std::mutex> lk(tc::g_mu);
    return tc::g_err.c_str();
}

cudaError_t launch_gemm1_tc(const void* S, const void* W1p, const float* b1, void* Hid, int B, int T, int D, int F,
                            int Bcap, int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    tc::Args a{};
    a.N = F;
    a.K = D;
    a.ngroups = T;
    a.group_base = 0;
    a.group_stride = 1;
    a.M = B;
    a.a_group_rows = Bcap;
    a.bias = b1;
    a.hid = reinterpret_cast<__half*>(Hid);
    a.hid_tma = 1;
    a.hid_evict_first = hid_evict_first(B, T, F) ? 1 : 0;
    a.rows_cap = (long long)T * Bcap;
    a.err = err;
    a.timeout_ns = timeout_ns;
    RM_HOST_BOUNDS(B <= Bcap && D % tc::BK == 0 && F % tc::BK == 0 && S && W1p && b1 && Hid);
    RM_HOST_BOUNDS(((reinterpret_cast<uintptr_t>(S) | reinterpret_cast<uintptr_t>(W1p) | reinterpret_cast<uintptr_t>(Hid)) &
                    15u) == 0);
    return tc::run_dense<tc::EPI_GELU>(tc::pick_bn(F), S, (long long)T * Bcap, W1p, T, a, num_sms, s);
}

cudaError_t launch_gemm2_tc(const void* Hid, const void* W2p, const float* b2, const void* S, void* Z,
                            float2* stats, int B, int T, int D, int F, int Bcap, int num_sms, int* err,
                            unsigned long long timeout_ns, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    const int bn = gemm2_bn(D);
    if (bn == 0) return cudaErrorNotSupported;
    tc::Args a{};
    a.N = D;
    a.K = F;
    a.ngroups = T;
    a.group_base = 0;
    a.group_stride = 1;
    a.M = B;
    a.a_group_rows = Bcap;
    a.bias = b2;
    a.resid = reinterpret_cast<const __half*>(S);
    a.z = reinterpret_cast<__half*>(Z);
    a.stats = stats;
    a.nchunk = D / (bn / 2);
    a.rows_cap = (long long)T * Bcap;
    a.err = err;
    a.timeout_ns = timeout_ns;
    RM_HOST_BOUNDS(B <= Bcap && D % tc::BK == 0 && F % tc::BK == 0 && Hid && W2p && b2 && S && Z && stats);
    RM_HOST_BOUNDS(((reinterpret_cast<uintptr_t>(Hid) | reinterpret_cast<uintptr_t>(W2p) | reinterpret_cast<uintptr_t>(S) |
                     reinterpret_cast<uintptr_t>(Z)) & 15u) == 0);
    return tc::run_dense<tc::EPI_RESID>(bn, Hid, (long long)T * Bcap, W2p, T, a, num_sms, s);
}

cudaError_t launch_moe_gemm1_tc(const void* Sg, long long rows_total, const void* W1p, const float* b1, void* Hm,
                                int groups, int D, int Fe, const int* g_count, const int* g_off,
                                const int* tile_prefix, const int* tile_prefix256, int num_sms, int* err,
                                unsigned long long timeout_ns, cudaStream_t s) {
    tc::Args a{};
    a.N = Fe;
    a.K = D;
    a.ngroups = groups;
    a.group_base = 0;
    a.group_stride = 1;
    a.g_count = g_count;
    a.g_off = g_off;
    a.tile_prefix = tile_prefix;
    a.bias = b1;
    a.hid = reinterpret_cast<__half*>(Hm);
    a.rows_cap = rows_total;
    a.err = err;
    a.timeout_ns = timeout_ns;
    RM_HOST_BOUNDS(D % tc::BK == 0 && Fe % tc::BK == 0 && Sg && W1p && b1 && Hm && g_count && g_off && tile_prefix);
    if (tile_prefix256 && tc::pick_bn(Fe) >= 128) {     // CTA-pair tiles over 256-row tiles
        a.tile_prefix = tile_prefix256;
        return tc::run_pair_bn<tc::EPI_GELU, 8>(tc::pick_bn(Fe), tc::use_ksub2(D, tc::EPI_GELU), Sg, rows_total,
                                                W1p, groups, a, num_sms, s);
    }
    return tc::run_bn<tc::EPI_GELU>(tc::pick_bn(Fe), Sg, rows_total, W1p, groups, a, num_sms, s);
}

cudaError_t launch_moe_gemm2_tc(const void* Hm, long long rows_total, const void* W2p, const float* b2, void* Y,
                                int groups, int D, int Fe, const int* g_count, const int* g_off,
                                const int* tile_prefix, const int* tile_prefix256, const float* row_gate,
                                int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    tc::Args a{};
    a.N = D;
    a.K = Fe;
    a.ngroups = groups;
    a.group_base = 0;
    a.group_stride = 1;
    a.g_count = g_count;
    a.g_off = g_off;
    a.tile_prefix = tile_prefix;
    a.bias = b2;
    a.hid = reinterpret_cast<__half*>(Y);
    a.row_gate = row_gate;
    a.rows_cap = rows_total;
    a.err = err;
    a.timeout_ns = timeout_ns;
    RM_HOST_BOUNDS(D % tc::BK == 0 && Fe % tc::BK == 0 && Hm && W2p && b2 && Y && row_gate && g_count && g_off);
    if (tile_prefix256 && tc::pick_bn(D) >= 128) {      // CTA-pair tiles over 256-row tiles
        a.tile_prefix = tile_prefix256;
        return tc::run_pair_bn<tc::EPI_GATED, 8>(tc::pick_bn(D), tc::use_ksub2(Fe, tc::EPI_GATED), Hm, rows_total,
                                                 W2p, groups, a, num_sms, s);
    }
    return tc::run_bn<tc::EPI_GATED>(tc::pick_bn(D), Hm, rows_total, W2p, groups, a, num_sms, s);
}

}  // namespace rm
