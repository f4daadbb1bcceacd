// UniMixing kernels ("UniMixer: A Unified Architecture for Scaling Laws in
// Recommendation Systems", section 4.3): the Sinkhorn-Knopp constraint of the
// mixing weights (Eq. 15), the per-block local step h_j = x_j WB_j (Eq. 13)
// and, after the global step WG H on the tensor cores (stored straight into
// the sample-major layout by its epilogue), the residual + LN1 that feeds the
// per-token FFN.
//
// All three are memory-bound or tiny: the local step reads each sample once
// and writes H once (bs^2 multiply-adds per block of bs values, packed fp32x2
// FMAs on a bs x bs weight tile in shared memory); the row kernel reads X and
// Y once, contiguously, and writes S once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <type_traits>

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

// Blocks for a grid-stride loop over `work` items (capped: the loops stride).
int grid_of(long long work, int threads) {
    long long g = (work + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > 4096) g = 4096;
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

// bs % 8 == 0, bs <= 64.  CTA (sample tile, block j): WB_j (float32) and the
// tile's x_j rows in shared memory, each x stored twice as an (x, x) pair so
// that one 8-byte load feeds the packed fp32x2 FMAs.  Thread (sg, rg) computes
// samples sg + k SG (k < 8) x columns 8 rg .. 8 rg + 7: per s, 8 pair loads,
// two 16-byte weight loads and 32 packed FMAs (64 multiply-adds).  A warp's
// stores for one k cover consecutive samples' contiguous bs-wide runs of H's
// row j.  The x rows are bs + 1 pairs apart (an odd stride: the sample groups
// of a warp read distinct banks).
template <typename Tx, typename Top>
__global__ void __launch_bounds__(128)
unimix_local_kernel(const Tx* __restrict__ X, long long x_stride, const float* __restrict__ WB, Top* __restrict__ H,
                    int B, int bs, long long Npitch, long long Npad) {
    constexpr int SPT = 8;
    extern __shared__ float4 smem4[];
    float* smem = reinterpret_cast<float*>(smem4);
    const int j = blockIdx.y;
    const int rq = bs >> 3;
    const int SG = blockDim.x / rq;
    const int SB = SG * SPT;
    const int ldx = bs + 1;                       // in pairs
    float* sW = smem;                             // [bs][bs]
    float2* sX = reinterpret_cast<float2*>(smem + bs * bs);   // [SB][bs + 1] pairs (x, x)
    const float* wsrc = WB + (size_t)j * bs * bs;
    for (int e = threadIdx.x; e < bs * bs; e += blockDim.x) sW[e] = wsrc[e];
    const long long b0 = (long long)blockIdx.x * SB;
    constexpr int VE = 16 / (int)sizeof(Tx);     // values per 16-byte load (bs % VE == 0)
    const int nseg = bs / VE;
    for (int e = threadIdx.x; e < SB * nseg; e += blockDim.x) {
        const int bb = e / nseg, s0 = (e - bb * nseg) * VE;
        const long long b = b0 + bb;
        float2* dst = sX + bb * ldx + s0;
        if (b < B) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(X + b * x_stride + (long long)j * bs + s0));
            const Tx* pv = reinterpret_cast<const Tx*>(&v);
#pragma unroll
            for (int u = 0; u < VE; ++u) {
                const float x = XLoad<Tx>::at(pv + u);
                dst[u] = make_float2(x, x);
            }
        } else {
#pragma unroll
            for (int u = 0; u < VE; ++u) dst[u] = make_float2(0.f, 0.f);
        }
    }
    __syncthreads();
    const int rg = threadIdx.x % rq, sg = threadIdx.x / rq;
    if (sg < SG) {
        uint64_t acc[SPT][4];
#pragma unroll
        for (int k = 0; k < SPT; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[k][q] = 0ull;
        const float2* xs = sX + sg * ldx;
        for (int s = 0; s < bs; ++s) {
            const float4 wa = *reinterpret_cast<const float4*>(sW + s * bs + 8 * rg);
            const float4 wb = *reinterpret_cast<const float4*>(sW + s * bs + 8 * rg + 4);
            const uint64_t w0 = f2_pack(wa.x, wa.y), w1 = f2_pack(wa.z, wa.w);
            const uint64_t w2 = f2_pack(wb.x, wb.y), w3 = f2_pack(wb.z, wb.w);
#pragma unroll
            for (int k = 0; k < SPT; ++k) {
                const uint64_t xv = *reinterpret_cast<const uint64_t*>(xs + (size_t)SG * k * ldx + s);
                acc[k][0] = f2_fma(xv, w0, acc[k][0]);
                acc[k][1] = f2_fma(xv, w1, acc[k][1]);
                acc[k][2] = f2_fma(xv, w2, acc[k][2]);
                acc[k][3] = f2_fma(xv, w3, acc[k][3]);
            }
        }
        Top* hrow = H + (size_t)j * Npitch;
#pragma unroll
        for (int k = 0; k < SPT; ++k) {
            const long long b = b0 + sg + SG * k;
            if (b < B) {
                float v[8];
                f2_unpack(acc[k][0], v[0], v[1]);
                f2_unpack(acc[k][1], v[2], v[3]);
                f2_unpack(acc[k][2], v[4], v[5]);
                f2_unpack(acc[k][3], v[6], v[7]);
                store4(hrow + b * bs + 8 * rg, v[0], v[1], v[2], v[3]);
                store4(hrow + b * bs + 8 * rg + 4, v[4], v[5], v[6], v[7]);
            }
        }
    }
    if (blockIdx.x == 0) {
        Top* hrow = H + (size_t)j * Npitch;
        for (long long n = (long long)B * bs + threadIdx.x; n < Npad; n += blockDim.x) hrow[n] = from_f32<Top>(0.f);
    }
}

// ---------------------------------------------------------------------------
// Local step on the tensor cores (warp-level mma.sync m16n8k16, fp16
// operands, fp32 accumulate): 2-byte inputs, BS a multiple of 16 up to 64.
// A warp keeps WB_j's fragments (BS / 16 k-steps x BS / 8 column tiles, from
// the transposed fp16 copy WBt[j][r][s]) in registers for its block j and
// streams tiles of 16 samples: A fragments straight from X (rows b, columns
// j BS + k; bf16 inputs converted to fp16, exact for every bf16 value of
// magnitude 2^-14 .. 65504), the 16 x BS result to H's row j as fp16 pairs.
// fp16 rather than bf16 weights: near-uniform (high-temperature) weights
// average the signal down over BS terms but not the weights' rounding, which
// at bf16's 8 significant bits reached 2.3e-2 of the output's rms at the 1B
// shape.  The step is bound by reading X and writing H; the products are a
// few percent of the tensor-core time.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two packed 16-bit inputs -> a packed fp16 pair.
template <typename Tin> __device__ __forceinline__ uint32_t to_f16x2(uint32_t v);
template <> __device__ __forceinline__ uint32_t to_f16x2<__half>(uint32_t v) { return v; }
template <> __device__ __forceinline__ uint32_t to_f16x2<__nv_bfloat16>(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

constexpr int kMmaWarps = 4;
constexpr int kMmaTilesPerWarp = 8;      // 16-sample tiles per warp per CTA (the fragments of W_B^j are loaded once per warp)

// K and N are permuted inside each 16 x BS tile so that a lane's operands and
// results are contiguous in memory: lane (g, c) holds, for its rows g and
// g + 8, the physical input columns [4 KS c, 4 KS (c + 1)) -- in k-step ks the
// fragment slots a0/a1 take columns 4 KS c + 4 ks + {0, 1} and a2/a3 take
// + {2, 3} -- and writes the physical output columns [2 NT c, 2 NT (c + 1)),
// n-tile nt's pair at 2 NT c + 2 nt.  The B fragments read W_B^j under the same
// two maps (logical column n = 8 nt + g of an n-tile is physical column
// 2 NT (g >> 1) + 2 nt + (g & 1)), so every output is the sum over the same k
// of the same products.  A lane then loads KS 8-byte words per row and stores
// NT / 2 8-byte words per row, and the next tile's words are loaded before the
// current tile's products.
template <typename Tin, int BS>
__global__ void __launch_bounds__(32 * kMmaWarps)
unimix_local_mma_kernel(const Tin* __restrict__ X, long long x_stride, const __half* __restrict__ WBt,
                        __half* __restrict__ H, int B, long long Npitch, long long Npad) {
    constexpr int KS = BS / 16, NT = BS / 8;
    static_assert(NT % 2 == 0, "output words of two n-tiles");
    const int j = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // B fragments: B[k][n] = WB_j[k][n] = WBt[j][n][k], physical k and n as above
    uint32_t bf[KS][NT][2];
    const __half* w = WBt + (size_t)j * BS * BS;
    const int ncol0 = (g >> 1) * 2 * NT + (g & 1);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const __half* row = w + (size_t)(ncol0 + 2 * nt) * BS + 4 * KS * c + 4 * ks;
            bf[ks][nt][0] = __ldg(reinterpret_cast<const uint32_t*>(row));
            bf[ks][nt][1] = __ldg(reinterpret_cast<const uint32_t*>(row + 2));
        }
    __half* hrow = H + (size_t)j * Npitch;
    const long long tile0 = ((long long)blockIdx.x * kMmaWarps + warp) * kMmaTilesPerWarp;
    // this lane's words of a tile: rows b0 + g and b0 + g + 8, KS 8-byte words each
    auto load_tile = [&](long long b0, uint2 (&x0w)[KS], uint2 (&x1w)[KS]) {
        const long long r0 = b0 + g, r1 = b0 + g + 8;
        const Tin* x0 = X + r0 * x_stride + (long long)j * BS + 4 * KS * c;
        const Tin* x1 = X + r1 * x_stride + (long long)j * BS + 4 * KS * c;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            x0w[ks] = r0 < B ? __ldg(reinterpret_cast<const uint2*>(x0) + ks) : make_uint2(0u, 0u);
            x1w[ks] = r1 < B ? __ldg(reinterpret_cast<const uint2*>(x1) + ks) : make_uint2(0u, 0u);
        }
    };
    uint2 n0w[KS], n1w[KS];
    if (tile0 * 16 < B) load_tile(tile0 * 16, n0w, n1w);
#pragma unroll 1
    for (int it = 0; it < kMmaTilesPerWarp; ++it) {
        const long long b0 = (tile0 + it) * 16;
        if (b0 >= B) break;
        uint2 x0w[KS], x1w[KS];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            x0w[ks] = n0w[ks];
            x1w[ks] = n1w[ks];
        }
        if (it + 1 < kMmaTilesPerWarp && b0 + 16 < B) load_tile(b0 + 16, n0w, n1w);
        uint32_t af[KS][4];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            af[ks][0] = to_f16x2<Tin>(x0w[ks].x);
            af[ks][1] = to_f16x2<Tin>(x1w[ks].x);
            af[ks][2] = to_f16x2<Tin>(x0w[ks].y);
            af[ks][3] = to_f16x2<Tin>(x1w[ks].y);
        }
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], af[ks], bf[ks][nt][0], bf[ks][nt][1]);
        const long long r0 = b0 + g, r1 = b0 + g + 8;
        uint2* o0 = reinterpret_cast<uint2*>(hrow + r0 * BS + 2 * NT * c);
        uint2* o1 = reinterpret_cast<uint2*>(hrow + r1 * BS + 2 * NT * c);
#pragma unroll
        for (int m = 0; m < NT / 2; ++m) {
            if (r0 < B)
                o0[m] = make_uint2(pack_f16x2(acc[2 * m][0], acc[2 * m][1]), pack_f16x2(acc[2 * m + 1][0], acc[2 * m + 1][1]));
            if (r1 < B)
                o1[m] = make_uint2(pack_f16x2(acc[2 * m][2], acc[2 * m][3]), pack_f16x2(acc[2 * m + 1][2], acc[2 * m + 1][3]));
        }
    }
    if (blockIdx.x == 0) {
        for (long long n = (long long)B * BS + threadIdx.x; n < Npad; n += blockDim.x) hrow[n] = __float2half_rn(0.f);
    }
}

// ---------------------------------------------------------------------------
// The same local step with the samples staged in shared memory by bulk copies
// (the same products in the same order as unimix_local_mma_kernel, so the same
// bits), for a deep, register-free read pipeline and whole-line writes.
//
// Work item: a group of kLsJ consecutive blocks j and 16 consecutive samples.
// Each CTA takes a contiguous run of items in group-major order, so its warps
// reload their W_B^j fragments only when the group changes.  A producer warp
// fills up to STAGES items ahead: per sample row one 1-D bulk copy of the
// group's kLsJ BS contiguous values (a 768-byte run at BS = 48), into a row
// pitch padded so that the 8-byte fragment loads of a half-warp fall on
// distinct banks (BS = 16 and 48; 2-way at 32 and 64).  Compute warp w takes
// block kLsJ g + w of every item of group g: A fragments from the staged rows
// under the K permutation above, the products, then the 16 x BS fp16 result
// into a per-warp staging buffer (two, alternating) and one bulk store into
// H's row j, where the 16 samples' BS values are contiguous.
// ---------------------------------------------------------------------------
// 1-D bulk copy shared -> global (both 16-byte aligned, size a multiple of 16)
// in the thread's current bulk async group.
__device__ __forceinline__ void bulk_copy_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes)
                 : "memory");
}

constexpr int kLsJ = 8;          // blocks per group = compute warps per CTA
constexpr int kLsRows = 16;      // samples per item (one m16 tile)

template <int BS>
struct LsCfg {
    static constexpr int ROW_BYTES = kLsJ * BS * 2;
    // row pitch = 24 (BS = 48) or 8 (BS = 16) 4-byte words mod 32
    static constexpr int PAD = BS == 48 ? 96 : (BS == 16 ? 32 : 16);
    static constexpr int PITCH = (ROW_BYTES + 127) / 128 * 128 + PAD;
    static constexpr int STAGE_BYTES = kLsRows * PITCH;
    static constexpr int OUT_BYTES = kLsRows * BS * 2;   // one warp's 16 x BS result
    static constexpr int STAGES = BS <= 48 ? 6 : 4;
    static constexpr int OUT_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = OUT_OFF + kLsJ * 2 * OUT_BYTES;
    static constexpr int SMEM = BAR_OFF + 2 * STAGES * 8 + 16;
    static constexpr int THREADS = 32 * (kLsJ + 1);
    static constexpr int MIN_BLOCKS = BS <= 48 ? 2 : 1;
    static_assert(PITCH % 16 == 0 && OUT_OFF % 16 == 0 && OUT_BYTES % 16 == 0, "bulk-copy alignment");
    static_assert(MIN_BLOCKS * (SMEM + 1024) <= 228 * 1024, "shared memory per SM");
};

template <typename Tin, int BS>
__global__ void __launch_bounds__(LsCfg<BS>::THREADS, LsCfg<BS>::MIN_BLOCKS)
unimix_local_staged_kernel(const Tin* __restrict__ X, long long x_stride, const __half* __restrict__ WBt,
                           __half* __restrict__ H, int B, int nb, long long Npitch, long long Npad, int* err,
                           unsigned long long timeout_ns) {
    using C = LsCfg<BS>;
    constexpr int KS = BS / 16, NT = BS / 8;
    extern __shared__ __align__(128) uint8_t ls_smem[];
    const uint32_t sbase = smem_u32(ls_smem);
    volatile int* abort = reinterpret_cast<volatile int*>(ls_smem + C::BAR_OFF + 2 * C::STAGES * 8);
    auto full = [&](int s) { return sbase + (uint32_t)C::BAR_OFF + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return sbase + (uint32_t)C::BAR_OFF + 8u * (uint32_t)(C::STAGES + s); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = (nb + kLsJ - 1) / kLsJ;
    const int ntiles = (B + kLsRows - 1) / kLsRows;
    const int items = ngroups * ntiles;   // < 2^31 (checked by the launcher)
    const int i0 = (int)((long long)items * blockIdx.x / gridDim.x);
    const int i1 = (int)((long long)items * (blockIdx.x + 1) / gridDim.x);
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kLsJ * 32);
        }
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kLsJ) {
        // ---- producer ----
        int i = i0;
        for (; i < i1; ++i) {
            const int n = i - i0;
            const int s = n % C::STAGES;
            const uint32_t ph = (uint32_t)(n / C::STAGES) & 1u;
            if (n >= C::STAGES && !mbar_wait_bounded(empty(s), ph ^ 1u, abort, err, timeout_ns)) break;
            const int jg = i / ntiles, bt = i - jg * ntiles;
            const int jv = min(kLsJ, nb - jg * kLsJ);
            const int b0 = bt * kLsRows, rows = min(kLsRows, B - b0);
            const uint32_t bytes = (uint32_t)jv * BS * 2u;
            if (lane == 0) mbar_arrive_expect_tx(full(s), (uint32_t)rows * bytes);
            __syncwarp();
            // (bounds-checked build: a skipped copy leaves the stage short, and the
            // compute warps' bounded wait then ends the launch with an error)
            if (lane < rows && RM_IN_BOUNDS(b0 + lane < B && (long long)jg * kLsJ * BS + jv * BS <= x_stride, err))
                bulk_copy_g2s(sbase + (uint32_t)s * C::STAGE_BYTES + (uint32_t)lane * C::PITCH,
                              X + (long long)(b0 + lane) * x_stride + (long long)jg * kLsJ * BS, bytes, full(s));
        }
        // The CTA may exit only after the copies it issued have landed.  The
        // compute warps wait for every stage they use; after an abort some are
        // not used, so wait (bounded, whatever the abort flag) on the last
        // fill of each stage.
        const int issued = i - i0;
        if (lane == 0) {
            for (int n = issued - 1; n >= 0 && n >= issued - C::STAGES; --n) {
                const int s = n % C::STAGES;
                const uint32_t ph = (uint32_t)(n / C::STAGES) & 1u;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(full(s), ph) && globaltimer_ns() - t0 < timeout_ns) {
                }
            }
        }
        return;
    }

    // ---- compute warp: block j = kLsJ g + warp of each item of group g ----
    const int g = lane >> 2, c = lane & 3;
    const int ncol0 = (g >> 1) * 2 * NT + (g & 1);
    uint32_t bf[KS][NT][2];
    int cur_jg = -1;
    int sbuf = 0;
    const int obase = C::OUT_OFF + warp * 2 * C::OUT_BYTES;
    for (int i = i0; i < i1; ++i) {
        const int n = i - i0;
        const int s = n % C::STAGES;
        const uint32_t ph = (uint32_t)(n / C::STAGES) & 1u;
        const int jg = i / ntiles, bt = i - jg * ntiles;
        const int j = jg * kLsJ + warp;
        const bool active = j < nb;
        if (active && jg != cur_jg) {
            // B[k][n] = WB_j[k][n] = WBt[j][n][k], physical k and n as in unimix_local_mma_kernel
            const __half* w = WBt + (size_t)j * BS * BS;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const __half* row = w + (size_t)(ncol0 + 2 * nt) * BS + 4 * KS * c + 4 * ks;
                    bf[ks][nt][0] = __ldg(reinterpret_cast<const uint32_t*>(row));
                    bf[ks][nt][1] = __ldg(reinterpret_cast<const uint32_t*>(row + 2));
                }
            cur_jg = jg;
        }
        if (!mbar_wait_bounded(full(s), ph, abort, err, timeout_ns)) break;
        float acc[NT][4];
        if (active) {
            const uint8_t* r0 = ls_smem + s * C::STAGE_BYTES + g * C::PITCH + warp * BS * 2 + 8 * KS * c;
            const uint8_t* r1 = r0 + 8 * C::PITCH;
            uint2 x0w[KS], x1w[KS];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                x0w[ks] = *reinterpret_cast<const uint2*>(r0 + 8 * ks);
                x1w[ks] = *reinterpret_cast<const uint2*>(r1 + 8 * ks);
            }
            uint32_t af[KS][4];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                af[ks][0] = to_f16x2<Tin>(x0w[ks].x);
                af[ks][1] = to_f16x2<Tin>(x1w[ks].x);
                af[ks][2] = to_f16x2<Tin>(x0w[ks].y);
                af[ks][3] = to_f16x2<Tin>(x1w[ks].y);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], af[ks], bf[ks][nt][0], bf[ks][nt][1]);
        }
        // Every lane releases the stage only after MMAs that take its loaded
        // words as operands have issued, i.e. after its shared-memory loads
        // have returned.  Arriving right after issuing the loads (by one lane
        // or by each) measured stage contents overwritten by the next copy
        // before some loads had read them.
        mbar_arrive(empty(s));
        if (!active) continue;
        const int b0 = bt * kLsRows, rows = min(kLsRows, B - b0);
        const int ob = obase + sbuf * C::OUT_BYTES;
        if (lane == 0) bulk_wait_group_read<1>();   // the store that last read this buffer
        __syncwarp();
        uint8_t* o0 = ls_smem + ob + g * BS * 2 + 4 * NT * c;
        uint8_t* o1 = o0 + 8 * BS * 2;
#pragma unroll
        for (int m = 0; m < NT / 2; ++m) {
            *reinterpret_cast<uint2*>(o0 + 8 * m) =
                make_uint2(pack_f16x2(acc[2 * m][0], acc[2 * m][1]), pack_f16x2(acc[2 * m + 1][0], acc[2 * m + 1][1]));
            *reinterpret_cast<uint2*>(o1 + 8 * m) =
                make_uint2(pack_f16x2(acc[2 * m][2], acc[2 * m][3]), pack_f16x2(acc[2 * m + 1][2], acc[2 * m + 1][3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (RM_IN_BOUNDS((long long)b0 * BS + (long long)rows * BS <= Npitch, err))
                bulk_copy_s2g(H + (long long)j * Npitch + (long long)b0 * BS, sbase + (uint32_t)ob,
                              (uint32_t)rows * BS * 2u);
            bulk_commit_group();
        }
        sbuf ^= 1;
        if (bt == ntiles - 1 && RM_IN_BOUNDS(Npad <= Npitch, err)) {   // row j's padding columns
            __half* hrow = H + (long long)j * Npitch;
            for (long long q = (long long)B * BS + lane; q < Npad; q += 32) hrow[q] = __float2half_rn(0.f);
        }
    }
    if (lane == 0) bulk_wait_group<0>();
}

// WBt16[j][r][s] = fp16(WB[j][s][r]).
__global__ void pack_wb_kernel(const float* __restrict__ WB, __half* __restrict__ WBt16, int nb, int bs) {
    const long long total = (long long)nb * bs * bs;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long j = idx / ((long long)bs * bs);
        const int rem = (int)(idx - j * bs * bs);
        const int r = rem / bs, s = rem - r * bs;
        const float v = WB[(size_t)j * bs * bs + (size_t)s * bs + r];
        WBt16[idx] = __float2half_rn(v);
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
// Residual + LN1 after the global step, one warp per (b, t) row of D values:
// S[t][b][:] = LN1(X[b][t][:] + Y[b][t][:]) in the operand type, token-major.
// Y is the global product in the sample-major layout (operand type).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&o)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(h[u]);
        o[2 * u] = f.x;
        o[2 * u + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const __half* p, float (&o)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 f = __half22float2(h[u]);
        o[2 * u] = f.x;
        o[2 * u + 1] = f.y;
    }
}

// 2-byte types, D = 256 NG: lane l holds values 256 k + 8 l .. + 7 of the row.
template <typename Tx, int NG>
__global__ void __launch_bounds__(256)
unimix_ln1_vec_kernel(const Tx* __restrict__ X, const __half* __restrict__ Y, __half* __restrict__ S,
                      const float* __restrict__ g1, const float* __restrict__ be1, int B, int T, int D, int Bcap,
                      float eps) {
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * T;
    for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((long long)gridDim.x * blockDim.x) >> 5) {
        const long long b = row / T;
        const int t = (int)(row - b * T);
        float v[NG][8];
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            const int d = 256 * k + 8 * lane;
            float x[8];
            load8(X + row * D + d, x);
            load8(Y + row * D + d, v[k]);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                v[k][u] += x[u];
                sum += v[k][u];
            }
        }
        const float mean = warp_sum(sum) / (float)D;
        float sq = 0.f;
#pragma unroll
        for (int k = 0; k < NG; ++k)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float e = v[k][u] - mean;
                sq += e * e;
            }
        const float rstd = rsqrtf(warp_sum(sq) / (float)D + eps);
        __half* srow = S + ((size_t)t * Bcap + b) * D;
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            const int d = 256 * k + 8 * lane;
            const float4 ga = __ldg(reinterpret_cast<const float4*>(g1 + d));
            const float4 gb = __ldg(reinterpret_cast<const float4*>(g1 + d + 4));
            const float4 ba = __ldg(reinterpret_cast<const float4*>(be1 + d));
            const float4 bb = __ldg(reinterpret_cast<const float4*>(be1 + d + 4));
            const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
            const float be[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
            uint4 w;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                pw[u] = pack_f16x2(fmaf((v[k][2 * u] - mean) * rstd, gg[2 * u], be[2 * u]),
                                   fmaf((v[k][2 * u + 1] - mean) * rstd, gg[2 * u + 1], be[2 * u + 1]));
            *reinterpret_cast<uint4*>(srow + d) = w;
        }
    }
}

// Any D <= 32 NI and type: lane l holds values l + 32 k.
template <typename Tx, typename Top, int NI>
__global__ void __launch_bounds__(256)
unimix_ln1_kernel(const Tx* __restrict__ X, const Top* __restrict__ Y, Top* __restrict__ S,
                  const float* __restrict__ g1, const float* __restrict__ be1, int B, int T, int D, int Bcap,
                  float eps) {
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * T;
    for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((long long)gridDim.x * blockDim.x) >> 5) {
        const long long b = row / T;
        const int t = (int)(row - b * T);
        float v[NI];
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int d = lane + 32 * k;
            v[k] = 0.f;
            if (d < D) {
                v[k] = to_f32(Y[row * D + d]) + XLoad<Tx>::at(X + row * D + d);
                sum += v[k];
            }
        }
        const float mean = warp_sum(sum) / (float)D;
        float sq = 0.f;
#pragma unroll
        for (int k = 0; k < NI; ++k)
            if (lane + 32 * k < D) {
                const float e = v[k] - mean;
                sq += e * e;
            }
        const float rstd = rsqrtf(warp_sum(sq) / (float)D + eps);
        Top* srow = S + ((size_t)t * Bcap + b) * D;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int d = lane + 32 * k;
            if (d < D) srow[d] = from_f32<Top>(fmaf((v[k] - mean) * rstd, g1[d], be1[d]));
        }
    }
}

template <typename Top, typename Tout>
__global__ void convert_kernel(const Top* __restrict__ in, Tout* __restrict__ out, long long n) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        out[i] = from_f32<Tout>(to_f32(in[i]));
}

int rows_grid(long long rows, int num_sms) {
    long long grid = (rows + 7) / 8;
    if (grid > (long long)num_sms * 16) grid = (long long)num_sms * 16;
    return grid < 1 ? 1 : (int)grid;
}

template <typename Tx, typename Top>
cudaError_t launch_ln1_t(const void* X, const void* Y, void* S, const float* g1, const float* be1, int B, int T,
                         int D, int Bcap, float eps, int num_sms, cudaStream_t s) {
    const int grid = rows_grid((long long)B * T, num_sms);
    if constexpr (sizeof(Tx) == 2 && std::is_same<Top, __half>::value) {
        if (D % 256 == 0 && D <= 1536) {
#define RM_LN1V(NG)                                                                                            \
    unimix_ln1_vec_kernel<Tx, NG><<<grid, 256, 0, s>>>((const Tx*)X, (const __half*)Y, (__half*)S, g1, be1, B, T, \
                                                       D, Bcap, eps)
            switch (D / 256) {
                case 1: RM_LN1V(1); break;
                case 2: RM_LN1V(2); break;
                case 3: RM_LN1V(3); break;
                case 4: RM_LN1V(4); break;
                case 5: RM_LN1V(5); break;
                default: RM_LN1V(6); break;
            }
#undef RM_LN1V
            return cudaGetLastError();
        }
    }
#define RM_LN1(NI)                                                                                          \
    unimix_ln1_kernel<Tx, Top, NI><<<grid, 256, 0, s>>>((const Tx*)X, (const Top*)Y, (Top*)S, g1, be1, B, T, D, \
                                                        Bcap, eps)
    const int ni = (D + 31) / 32;
    if (ni <= 8) RM_LN1(8);
    else if (ni <= 16) RM_LN1(16);
    else if (ni <= 32) RM_LN1(32);
    else if (ni <= 48) RM_LN1(48);
    else return cudaErrorNotSupported;
#undef RM_LN1
    return cudaGetLastError();
}

template <typename Tx, typename Top>
cudaError_t launch_local_t(const void* X, long long x_stride, const float* WB, void* H, int B, int nb, int bs,
                           long long Npitch, long long Npad, cudaStream_t s) {
    constexpr int VE = 16 / (int)sizeof(Tx);
    if (bs % 8 == 0 && bs % VE == 0 && bs <= 64) {
        const int rq = bs / 8;
        const int SG = 128 / rq;
        const int threads = SG * rq;
        const int SB = SG * 8;
        const size_t smem = (size_t)bs * bs * sizeof(float) + (size_t)SB * (bs + 1) * sizeof(float2);
        auto k = unimix_local_kernel<Tx, Top>;
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

template <typename Tin>
cudaError_t launch_mma_t(const void* X, long long x_stride, const void* WBt16, void* H, int B, int nb, int bs,
                         long long Npitch, long long Npad, cudaStream_t s) {
    const long long per_cta = 16LL * kMmaWarps * kMmaTilesPerWarp;
    const dim3 grid((unsigned)((B + per_cta - 1) / per_cta), (unsigned)nb);
#define RM_MMA(BSV)                                                                                          \
    unimix_local_mma_kernel<Tin, BSV><<<grid, 32 * kMmaWarps, 0, s>>>((const Tin*)X, x_stride, (const __half*)WBt16, \
                                                                       (__half*)H, B, Npitch, Npad)
    switch (bs) {
        case 16: RM_MMA(16); break;
        case 32: RM_MMA(32); break;
        case 48: RM_MMA(48); break;
        case 64: RM_MMA(64); break;
        default: return cudaErrorNotSupported;
    }
#undef RM_MMA
    return cudaGetLastError();
}

bool unimix_local_mma_ok(int bs) { return bs == 16 || bs == 32 || bs == 48 || bs == 64; }

// RM_UNIMIX_LOCAL=regs in the environment keeps the register-prefetch local
// step (a tuning switch: the same products, the same bits).
bool local_staged_enabled() {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_UNIMIX_LOCAL");
        env = (v && v[0] == 'r') ? 0 : 1;
    }
    return env == 1;
}

template <typename Tin, int BS>
cudaError_t launch_staged_bs(const void* X, long long x_stride, const void* WBt16, void* H, int B, int nb,
                             long long Npitch, long long Npad, int num_sms, int* err, unsigned long long timeout_ns,
                             cudaStream_t s) {
    using C = LsCfg<BS>;
    auto k = unimix_local_staged_kernel<Tin, BS>;
    cudaError_t attr = smem_attr_once((const void*)k, C::SMEM);
    if (attr != cudaSuccess) return attr;
    const long long items = (long long)((nb + kLsJ - 1) / kLsJ) * ((B + kLsRows - 1) / kLsRows);
    if (items >= (1LL << 31)) return cudaErrorNotSupported;
    const long long slots = (long long)C::MIN_BLOCKS * (num_sms > 0 ? num_sms : 1);
    const int grid = (int)(items < slots ? items : slots);
    k<<<grid, C::THREADS, C::SMEM, s>>>((const Tin*)X, x_stride, (const __half*)WBt16, (__half*)H, B, nb, Npitch,
                                         Npad, err, timeout_ns);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_staged_t(const void* X, long long x_stride, const void* WBt16, void* H, int B, int nb, int bs,
                            long long Npitch, long long Npad, int num_sms, int* err, unsigned long long timeout_ns,
                            cudaStream_t s) {
    switch (bs) {
        case 16: return launch_staged_bs<Tin, 16>(X, x_stride, WBt16, H, B, nb, Npitch, Npad, num_sms, err, timeout_ns, s);
        case 32: return launch_staged_bs<Tin, 32>(X, x_stride, WBt16, H, B, nb, Npitch, Npad, num_sms, err, timeout_ns, s);
        case 48: return launch_staged_bs<Tin, 48>(X, x_stride, WBt16, H, B, nb, Npitch, Npad, num_sms, err, timeout_ns, s);
        case 64: return launch_staged_bs<Tin, 64>(X, x_stride, WBt16, H, B, nb, Npitch, Npad, num_sms, err, timeout_ns, s);
        default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_unimix_pack_wb(const float* WB, void* WBt16, int nb, int bs, cudaStream_t s) {
    pack_wb_kernel<<<grid_of((long long)nb * bs * bs, 256), 256, 0, s>>>(WB, (__half*)WBt16, nb, bs);
    return cudaGetLastError();
}

cudaError_t launch_unimix_local(XType xt, Act act, const void* X, long long x_stride, const float* WB,
                                const void* WBt16, void* H, int B, int nb, int bs, long long Npitch, long long Npad,
                                int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act != Act::F32 && WBt16 && unimix_local_mma_ok(bs) && x_stride % 8 == 0) {
        // the staged kernel's bulk copies: 16-byte aligned rows in X and in H
        const bool aligned16 = ((uintptr_t)X % 16 == 0) && ((uintptr_t)H % 16 == 0) && Npitch % 8 == 0;
        if (aligned16 && local_staged_enabled() && xt != XType::F32) {
            RM_HOST_BOUNDS(Npitch >= (long long)B * bs && Npad <= Npitch && x_stride >= (long long)nb * bs);
            if (xt == XType::BF16)
                return launch_staged_t<__nv_bfloat16>(X, x_stride, WBt16, H, B, nb, bs, Npitch, Npad, num_sms, err,
                                                      timeout_ns, s);
            return launch_staged_t<__half>(X, x_stride, WBt16, H, B, nb, bs, Npitch, Npad, num_sms, err, timeout_ns, s);
        }
        if (xt == XType::BF16)
            return launch_mma_t<__nv_bfloat16>(X, x_stride, WBt16, H, B, nb, bs, Npitch, Npad, s);
        if (xt == XType::F16) return launch_mma_t<__half>(X, x_stride, WBt16, H, B, nb, bs, Npitch, Npad, s);
    }
    if (act == Act::F32) {
        if (xt != XType::F32) return cudaErrorInvalidValue;
        return launch_local_t<float, float>(X, x_stride, WB, H, B, nb, bs, Npitch, Npad, s);
    }
    if (xt == XType::BF16) return launch_local_t<__nv_bfloat16, __half>(X, x_stride, WB, H, B, nb, bs, Npitch, Npad, s);
    if (xt == XType::F16) return launch_local_t<__half, __half>(X, x_stride, WB, H, B, nb, bs, Npitch, Npad, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_unimix_ln1(XType xt, Act act, const void* X, const void* Y, void* S, const float* g1,
                              const float* be1, int B, int T, int D, int Bcap, float eps, int num_sms,
                              cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    if (act == Act::F32) {
        if (xt != XType::F32) return cudaErrorInvalidValue;
        return launch_ln1_t<float, float>(X, Y, S, g1, be1, B, T, D, Bcap, eps, num_sms, s);
    }
    if (xt == XType::BF16) return launch_ln1_t<__nv_bfloat16, __half>(X, Y, S, g1, be1, B, T, D, Bcap, eps, num_sms, s);
    if (xt == XType::F16) return launch_ln1_t<__half, __half>(X, Y, S, g1, be1, B, T, D, Bcap, eps, num_sms, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_unimix_out(Act act, const void* Y, void* out, bool out_f32, long long n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (act == Act::F32)
        return cudaMemcpyAsync(out, Y, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, s);
    if (out_f32)
        convert_kernel<__half, float><<<grid_of(n, 256), 256, 0, s>>>((const __half*)Y, (float*)out, n);
    else
        convert_kernel<__half, __nv_bfloat16><<<grid_of(n, 256), 256, 0, s>>>((const __half*)Y, (__nv_bfloat16*)out,
                                                                              n);
    return cudaGetLastError();
}

}  // namespace rm
