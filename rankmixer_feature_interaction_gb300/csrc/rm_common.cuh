// Shared device helpers for the RankMixer sm_103a kernels: element conversion,
// warp reductions, the LayerNorm statistic merge, and thin inline-PTX wrappers
// for mbarrier, TMA (cp.async.bulk.tensor) and tcgen05 (MMA, TMEM).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rm_internal.h"

namespace rm {

// ---------------------------------------------------------------------------
// Element conversion
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// fp16 stores saturate finite overflow at +-65504 (NaN stays NaN).  The
// tensor-core operands of the bf16 path are fp16: LN outputs are bounded by
// sqrt(D) max|gamma| + max|beta| and GELU outputs by their input, far inside
// fp16's range, and fp16 carries 3 more mantissa bits than bf16.
__device__ __forceinline__ float sat_f16(float x) { return fabsf(x) > 65504.f ? copysignf(65504.f, x) : x; }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(sat_f16(x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
// Two floats -> packed fp16x2 (lo in the low half), round to nearest, finite
// overflow saturated to +-65504 (NaN stays NaN): one cvt instruction.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// GELU in its exact form u * Phi(u), Phi(u) = (1 + erf(u / sqrt 2)) / 2
// ("RankMixer 详解（1）" section 4.1), branch-free.  The complementary error
// function of x = |u| / sqrt 2 >= 0 comes from Abramowitz & Stegun, Handbook
// of Mathematical Functions (1964), formula 7.1.26 (after Hastings):
//   1 - erf(x) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
//   t = 1 / (1 + p x),  |error in erf| <= 1.5e-7,
//   p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741,
//   -1.453152027, 1.061405429.
// With c = 1 - erf(x): Gelu(u) = u - u c / 2 for u >= 0 and u c / 2 for u < 0
// (no cancellation for negative u).  To save instructions the code works
// with x' = |u| sqrt(log2(e) / 2), so exp(-x^2) = 2^(-x'^2) and t = 1 / (1 + p' x')
// with p' = p / (sqrt 2 sqrt(log2(e) / 2)), and carries the 1/2 in the
// coefficients (ah_i = a_i / 2).  Reciprocal and 2^y use the MUFU unit.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float gelu_erf(float u) {
    constexpr float k1 = 0.8493218002880191f;     // sqrt(log2(e) / 2)
    constexpr float pp = 0.27273748087922245f;    // p / (sqrt(2) k1)
    constexpr float ah1 = 0.127414796f, ah2 = -0.142248368f, ah3 = 0.7107068705f, ah4 = -0.7265760135f,
                    ah5 = 0.5307027145f;
    const float xp = fabsf(u) * k1;
    const float t = rcp_approx(fmaf(pp, xp, 1.0f));
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, ah5, ah4), ah3), ah2), ah1);
    const float uc = u * (poly * ex2_approx(-xp * xp));   // u (1 - erf(|u| / sqrt 2)) / 2
    return u >= 0.0f ? u - uc : uc;
}

// The same GELU for two values at once, with the packed fp32x2 arithmetic of
// sm_100+ (one instruction per pair for add, multiply and fused multiply-add).
// Written as Gelu(u) = relu(u) - |u| c / 2 with c = 1 - erf(|u| / sqrt 2),
// which holds for both signs (u >= 0: u - u c / 2; u < 0: u c / 2), has no
// branch and no cancellation for negative u; relu(u) = (u + |u|) / 2 is exact.
// The coefficients carry the sign of -c / 2 so that the last step is one fma.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_splat(float x) { return f2_pack(x, x); }

// (Gelu(u0 + b0), Gelu(u1 + b1)) as a packed pair
__device__ __forceinline__ uint64_t gelu_erf_x2(uint64_t u, uint64_t b) {
    constexpr float k1 = 0.8493218002880191f;     // sqrt(log2(e) / 2)
    constexpr float pp = 0.27273748087922245f;    // p / (sqrt(2) k1)
    // -a_i / 2 (Abramowitz & Stegun 7.1.26)
    constexpr float nh1 = -0.127414796f, nh2 = 0.142248368f, nh3 = -0.7107068705f, nh4 = 0.7265760135f,
                    nh5 = -0.5307027145f;
    u = f2_add(u, b);
    const uint64_t a = u & 0x7fffffff7fffffffull;                   // |u|
    const uint64_t xp = f2_mul(a, f2_splat(k1));
    const uint64_t den = f2_fma(f2_splat(pp), xp, f2_splat(1.0f));
    float d0, d1;
    f2_unpack(den, d0, d1);
    const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
    uint64_t q = f2_fma(t, f2_splat(nh5), f2_splat(nh4));
    q = f2_fma(t, q, f2_splat(nh3));
    q = f2_fma(t, q, f2_splat(nh2));
    q = f2_fma(t, q, f2_splat(nh1));
    q = f2_mul(q, t);                                               // -c / (2 e)
    const uint64_t sq = f2_mul(xp, xp);
    float s0, s1;
    f2_unpack(sq, s0, s1);
    const uint64_t e = f2_pack(ex2_approx(-s0), ex2_approx(-s1));   // exp(-u^2 / 2)
    const uint64_t w = f2_mul(q, e);                                // -c / 2
    const uint64_t relu = f2_mul(f2_add(u, a), f2_splat(0.5f));
    return f2_fma(a, w, relu);
}

// Packed fp32 pair -> packed fp16 pair (saturating)
__device__ __forceinline__ uint32_t pack_f16x2_from_f2(uint64_t v) {
    float lo, hi;
    f2_unpack(v, lo, hi);
    return pack_f16x2(lo, hi);
}

// ---------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Merge per-chunk LayerNorm partials into the row's (mean, M2).  Each chunk c
// of width cw holds (mean_c, M2_c) with M2_c = sum over the chunk of
// (z - mean_c)^2.  Chan et al.'s pairwise update, written for equal chunk
// sizes:  mean = (1/nchunk) sum_c mean_c,  M2 = sum_c (M2_c + cw (mean_c - mean)^2).
// The sums run over c in order with explicit fused multiply-adds, so that every
// kernel that merges a row (the merge kernel, or a consumer that merges the
// partials itself) gets the same bits.
__device__ __forceinline__ float2 merge_chunks(const float2* __restrict__ st, int nchunk, int cw) {
    float s = 0.f;
    for (int c = 0; c < nchunk; ++c) s = __fadd_rn(s, st[c].x);
    const float mean = __fdiv_rn(s, (float)nchunk);
    float m2 = 0.f;
    for (int c = 0; c < nchunk; ++c) {
        const float2 v = st[c];
        const float d = __fsub_rn(v.x, mean);
        m2 = __fadd_rn(m2, __fmaf_rn(__fmul_rn((float)cw, d), d, v.y));
    }
    return make_float2(mean, m2);
}

// Row (mean, rstd) from nchunk partials (nchunk = 1: already merged).  Every
// lane of the calling warp returns the same values.
__device__ __forceinline__ void merge_row_stats(const float2* __restrict__ st, int nchunk, int cw, int D,
                                                float eps, int lane, float& mean, float& rstd) {
    (void)lane;
    const float2 v = nchunk == 1 ? st[0] : merge_chunks(st, nchunk, cw);
    mean = v.x;
    rstd = rsqrtf(v.y / (float)D + eps);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The forward-path kernels are launched with
// programmatic stream serialization (launch_k in rm_internal.h): such a kernel
// may start while the previous kernel of the stream is still running, so it
// calls pdl_wait() before its first access to anything earlier work on the
// stream wrote or still reads (it returns at once for a normal launch), and
// pdl_launch_next() to let the next kernel begin launching (its CTAs then
// take SMs as this kernel's CTAs leave them, and run their set-up).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Bounded waiting
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void latch_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Device-side guard of the bounds-checked debug build: true when the access
// may proceed; otherwise latches kDevErrBounds and the caller skips it.
__device__ __forceinline__ bool in_bounds(bool ok, int* err) {
    if (!ok) latch_error(err, kDevErrBounds);
    return ok;
}
#ifdef RM_DEBUG_BOUNDS
#define RM_IN_BOUNDS(cond, err) ::rm::in_bounds((cond), (err))
#else
#define RM_IN_BOUNDS(cond, err) true
#endif

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// timeout_ns of global time, or as soon as another role of the CTA has set
// *abort; on giving up it sets *abort, latches kDevErrTimeout and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  int* err, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort = 1;
                latch_error(err, kDevErrTimeout);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies, global -> shared), completion on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(const CUtensorMap* m, uint32_t dst, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16),
// completion counted in bytes on an mbarrier.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy / TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The same between the generic and the async proxy for global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}


// Tiled TMA store shared -> global (bulk async group), and its completion waits.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N committed bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit operands -> f32, both K-major.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when every previously issued tcgen05.mma of
// this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape, x32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load without the wait: the registers are valid only after
// tmem_wait_ld(), so a caller can compute on the previous chunk meanwhile.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 64 16-bit elements (128 B), 8-row swizzle atoms of
// 1024 B stacked along M/N (stride-byte-offset 1024), descriptor version 1,
// layout type 2 (SWIZZLE_128B).  The tile base must be 1024-byte aligned;
// stepping K by 16 elements inside the atom adds 32 B to the start address.
__device__ __forceinline__ uint64_t make_sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address      [0,14)
    d |= (uint64_t)(1u) << 16;                          // leading byte offset (unused for SW128 K-major) [16,30)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset [32,46)
    d |= (uint64_t)1u << 46;                            // descriptor version [46,48)
    d |= (uint64_t)2u << 61;                            // SWIZZLE_128B       [61,64)
    return d;
}

// Instruction descriptor for kind::f16: D f32, A and B fp16 (format 0), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.  A and B always share a type.
__host__ __device__ constexpr uint32_t make_idesc_f16_f32(int M, int N) {
    return (1u << 4)                        // D format: f32
         | (0u << 7)                        // A format: f16
         | (0u << 10)                       // B format: f16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}


// ---------------------------------------------------------------------------
// CTA pairs (clusters of 2) for tcgen05 cta_group::2
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// All threads of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly another CTA's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Tiled TMA load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA of the pair (cta_group::2).
__device__ __forceinline__ void tma_load_3d_pair(const CUtensorMap* m, uint32_t dst, uint32_t bar_cluster, int x, int y,
                                                 int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMA issued by the even CTA: D (M = 256 over both CTAs' TMEM, 128 lanes
// each) (+)= A (128 rows from each CTA's shared memory) x B^T (N/2 rows from each).
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at this shared offset in every CTA of cta_mask
// when all prior pair MMAs of this thread have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"(cta_mask)
        : "memory");
}

}  // namespace rm
