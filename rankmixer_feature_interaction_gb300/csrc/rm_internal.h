// Internal launcher interface between the C-ABI layer (rm_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rm {

// Caller-facing activation dtype of a context.  Internally a BF16 context
// keeps its GEMM operands (S, hidden activations, packed weights) in fp16
// ("operand" type); an F32 context keeps everything in float32.
enum class Act { F32 = 0, BF16 = 1 };

// Device error word values (latched with atomicCAS from 0).
constexpr int kDevErrTimeout = 5;
constexpr int kDevErrOther = 6;
constexpr int kDevErrBounds = 7;    // a device-side bounds guard of the debug build fired

// Bounds-checked debug build (compiled with -DRM_DEBUG_BOUNDS, library
// librankmixer_debug.so): the launchers check their sizes, strides and
// alignments against the buffers they describe before any launch, and the
// kernels guard their global-memory accesses with RM_IN_BOUNDS, which latches
// kDevErrBounds in the context's error word and skips the access.  In the
// normal build both compile to nothing.
#ifdef RM_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif
// Host-side launcher check of the debug build: a failed condition returns
// cudaErrorInvalidValue from the launcher with the condition's text recorded.
cudaError_t debug_bounds_fail(const char* what);
#define RM_HOST_BOUNDS(cond)                                                   \
    do {                                                                       \
        if (::rm::kDebugBounds && !(cond)) return ::rm::debug_bounds_fail(#cond); \
    } while (0)

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) acts on the current device:
// set it once per (kernel, device), so that a process driving several GPUs
// gets it on each.
cudaError_t smem_attr_once(const void* func, int bytes);
// Resident clusters of two CTAs of `func` on the current device at `smem`
// bytes per CTA and `threads` per CTA, cached per (kernel, device); falls back
// to half the SM count if the query fails.
int pair_occupancy_once(const void* func, int threads, int smem, int num_sms);

inline size_t act_size(Act a) { return a == Act::F32 ? 4 : 2; }
inline size_t op_size(Act a) { return a == Act::F32 ? 4 : 2; }

// Every device allocation of the library goes through these two: device_alloc
// counts live allocations and can be made to fail on purpose (a host-side
// injection for the failure-detection tests: RM_FAULT_INJECT=alloc:N in the
// environment, or rm_debug_fail_alloc), device_free releases (nullptr: no-op).
cudaError_t device_alloc(void** p, size_t bytes);
void device_free(void* p);

// Kernel launch with programmatic stream serialization (the kernel may begin
// while the stream's previous kernel finishes; it must call pdl_wait() before
// touching memory earlier work wrote or reads).  RM_PDL=0 in the environment
// turns the attribute off (ordinary stream order; the same results).
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

// Token-major workspace: element (t, b, j) of a [T][Bcap][W] buffer sits at
// (t * Bcap + b) * W + j.

struct MixLnArgs {
    // input: either X (sample-major [B][T][D], caller dtype) ...
    const void* X;
    // ... or the previous layer's pre-LN2 rows Z (token-major, operand type)
    // with per-row chunk statistics and that layer's LN2 affine, finalised in fp32.
    const void* Z;
    const float2* stats;
    const float* g2;
    const float* be2;
    // output S (token-major, operand type) and this layer's LN1 affine
    void* S;
    const float* g1;
    const float* be1;
    int B, T, D, q, Bcap, nchunk, cw;
    float eps;
    int* err;                        // device error word for bounded waits (nullable)
    unsigned long long timeout_ns;
    // test hook only (launch_mix_residual_debug): y = Mix(X) + X as float32,
    // token-major [T][Bcap][D], instead of S
    float* Ydbg;
    // staged 8-wide kernel: CTAs per sample (set by its launcher; 0 or 1: one)
    int rsplit;
};

// S = LN1(Mix(X) + X).
cudaError_t launch_mix_ln1(Act act, bool from_z, const MixLnArgs& a, int num_sms, cudaStream_t s);

// Test hook: the staged 8-wide mixing kernel's residual sum y = Mix(X) + X,
// written as float32 to a.Ydbg ([T][Bcap][D]) in place of LN1.  from_z: the
// source rows are fp16 token-major (a.Z) and the kernel's LN2 finalisation is
// the identity (mean 0, rstd 1, gamma 1, beta 0), so y is the fp16 sum of the
// two gathered fp16 values; otherwise a.X is bf16 sample-major and y is their
// float32 sum.  cudaErrorNotSupported for shapes the 8-wide kernel does not take.
cudaError_t launch_mix_residual_debug(bool from_z, const MixLnArgs& a, int num_sms, cudaStream_t s);

// X_out[b][t][:] = LN2(Z[t][b][:]) in the caller dtype (Z in the operand type),
// or in float32 when out_f32 (the same float32 values before any rounding).
cudaError_t launch_ln2_out(Act act, const void* Z, const float2* stats, const float* g2, const float* be2,
                           void* X_out, bool out_f32, int B, int T, int D, int Bcap, int nchunk, int cw, float eps,
                           int num_sms, cudaStream_t s);

// pooled[b][:] = (1/T) sum_t X_L[b][t][:] with X_L = LN2(Z) in float32; XL (optional)
// receives X_L sample-major, rounded to the caller dtype, or as float32 when xl_f32.
cudaError_t launch_pool(Act act, const void* Z, const float2* stats, const float* g2, const float* be2,
                        float* pooled, void* XL, bool xl_f32, int B, int T, int D, int Bcap, int nchunk, int cw,
                        float eps, int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s);

// Merge each row's nchunk chunk partials (GEMM2 epilogue) into (mean, M2) of the row.
cudaError_t launch_stats_finalize(const float2* part, float2* out, int B, int T, int Bcap, int nchunk, int cw,
                                  int num_sms, cudaStream_t s);

// (mean, M2) of each full row of Z (operand type; one chunk per row).
cudaError_t launch_rowstats(Act act, const void* Z, float2* stats, int B, int T, int D, int Bcap, int num_sms,
                            cudaStream_t s);

// Token-major operand-type [T][Bcap][D] -> sample-major caller-dtype [B][T][D]
// (float32 when out_f32: the operand values exactly).
cudaError_t launch_token_to_sample(Act act, const void* src, void* dst, bool out_f32, int B, int T, int D, int Bcap,
                                   cudaStream_t s);

// Y[b][h][t q + r] = X[b][t][h q + r] on raw element bits (esz 2 or 4).
cudaError_t launch_token_mix(const void* X, void* Y, int B, int T, int D, int H, int esz, cudaStream_t s);

// out[g][c][r] = op(in[g][r][c]) for G matrices of R x C: caller dtype in,
// operand type out (bf16 -> fp16 conversion for BF16 contexts).
cudaError_t launch_pack_transpose(Act act, const void* in, void* out, int G, int R, int C, cudaStream_t s);

// out[g][c][r] = in[g][r][c], float32.
cudaError_t launch_transpose_f32(const float* in, float* out, int G, int R, int C, cudaStream_t s);

// out[i] = float(in[i]) for n elements of the caller dtype.
cudaError_t launch_to_f32(Act act, const void* in, float* out, size_t n, cudaStream_t s);

// Test hook: out[i] = the GELU the GEMM epilogues use, applied to u[i].
cudaError_t launch_debug_gelu(const float* u, float* out, long long n, int form, cudaStream_t s);

// Test hook: bounded wait on a flag nothing sets; latches kDevErrTimeout.
cudaError_t launch_debug_wait(const int* flag, int* err, unsigned long long timeout_ns, cudaStream_t s);

// ---- per-token FFN GEMMs -------------------------------------------------
// GEMM1: Hid[t] = Gelu(S[t] W1_t + b1_t), GEMM2: Z[t] = Hid[t] W2_t + b2_t + S[t].
// Activations (and Z) token-major in the operand type, weights packed K-major:
// W1p [T][N=kD][K=D], W2p [T][N=D][K=kD].

cudaError_t launch_gemm1_simt(Act act, const void* S, const void* W1p, const float* b1, void* Hid, int B, int T,
                              int D, int F, int Bcap, cudaStream_t s);
cudaError_t launch_gemm2_simt(Act act, const void* Hid, const void* W2p, const float* b2, const void* S, void* Z,
                              int B, int T, int D, int F, int Bcap, cudaStream_t s);

// tcgen05 path (fp16 operands; BF16 contexts only).
bool tc_supported(int D, int F);
int tc_stats_chunk_width(int D);   // chunk width of the LN2 partial statistics written by GEMM2
cudaError_t launch_gemm1_tc(const void* S, const void* W1p, const float* b1, void* Hid, int B, int T, int D, int F,
                            int Bcap, int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s);
cudaError_t launch_gemm2_tc(const void* Hid, const void* W2p, const float* b2, const void* S, void* Z,
                            float2* stats, int B, int T, int D, int F, int Bcap, int num_sms, int* err,
                            unsigned long long timeout_ns, cudaStream_t s);

// Both FFN GEMMs of a dense layer in one launch (tensor-core CTA pairs, B >=
// 256 rows per token): the same results as launch_gemm1_tc + launch_gemm2_tc.
// dep_cnt: [T][ceil(Bcap / 256)] counters that only grow, dep_epoch the number
// of fused launches made on them before (both owned by the caller; zero the
// counters and the epoch together).  cudaErrorNotSupported when the shape or
// batch does not qualify (layer_tc_fusable).
bool layer_tc_fusable(int B, int D, int F);
cudaError_t launch_layer_tc(const void* S, const void* W1p, const float* b1, void* Hid, const void* W2p,
                            const float* b2, void* Z, float2* stats, int B, int T, int D, int F, int Bcap, int num_sms,
                            unsigned* dep_cnt, unsigned dep_epoch, int* err, unsigned long long timeout_ns,
                            cudaStream_t s);

// Set by the tensor-map encoder when the driver call fails (host-side message).
const char* tc_last_error();

}  // namespace rm
