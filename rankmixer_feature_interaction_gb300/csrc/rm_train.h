// Internal launcher interface of the block backward pass ("RankMixer 详解（1）"
// section 5.2).  Not part of the public ABI.
//
// Every GEMM of the backward pass, and the forward recompute it starts with,
// is a set of G independent per-token products
//     C_g[m][n] = sum_k A_g(m, k) B_g(n, k)      (fp32 accumulate)
// whose operands are either K-major (element (r, k) at r * inner + k) or
// MN-major (element (r, k) at k * inner + r), so weight gradients read the
// token-major activations [T][Bcap][W] and the caller-layout weights in place.
#pragma once

#include <cuda_runtime.h>

#include "rm_internal.h"

namespace rm {

// One operand of a grouped product.  K-major: inner = K, outer = the M (or N)
// rows; MN-major: inner = M (or N), outer = the K rows.  Rows at or past
// `outer` (and columns at or past `inner`) read as zero.  Group g starts
// gpitch elements after group g - 1.
struct TOperand {
    const void* ptr;
    int inner;
    int outer;
    long long gpitch;
    bool mn;
    long long ld = 0;       // elements between consecutive outer rows (0: inner)
};

// Operand precision.  float32 contexts run every product in float32.  bf16
// contexts run them on fp16 operands (11 significant bits) with float32
// accumulation: the recomputed activations S, Gelu(U), Gelu'(U) and Z are
// O(1) and the weights convert from bf16 exactly (apart from values below
// 2^-14 in magnitude); the two gradient operands dZ and dU carry a per-token
// power-of-two scale s_t that brings token t's largest |dZ| to 2^9, so
// gradients of any magnitude keep fp16's relative precision.  Products with a
// scaled operand multiply their accumulator by inv_scale[g] = 1 / s_g (exact).
//
// Epilogues.  Row m, column n of group g of C, and of the row-aligned inputs
// R / Gp, sit at g * c_gpitch + m * c_ld + n (c_ld = N unless set); rows
// m >= m_valid are not stored.
// "acc" below is the accumulator times inv_scale[g] where inv_scale is given.
enum TrainEpi {
    TE_GELU2 = 1,    // C0 = Gelu(acc + bias)  (operand type), C1 = Gelu'(acc + bias)  (aux type)
    TE_RESID = 2,    // C0 = acc + bias + R    (aux type; R operand type)
    TE_DGELU = 3,    // C0 = raw accumulator * Gp (operand type, stays in the scaled domain; Gp aux
                     //      type), plus column partial sums of acc * Gp
    TE_DRESID = 4,   // C0 = acc + R           (float; R float)
    TE_F32 = 5,      // C0 = acc               (float)
    TE_BIAS_IO = 6,  // C0 = acc + bias        (the context's caller dtype: bf16 or float)
    TE_F16 = 7,      // C0 = acc               (operand type: fp16, or float for float32 contexts)
    TE_F16T = 8,     // as TE_F16, stored for UniMixing's sample-major layout: column n = b um_bs + r
                     //      of row m goes to C0[b um_L + m um_bs + r], columns with b >= um_B are
                     //      dropped (um_bs a multiple of 8 on the tensor-core path)
};

struct TrainGemm {
    int G, M, N, K;
    int m_valid;
    TOperand a, b;
    long long c_gpitch;
    long long c_ld;         // elements between consecutive rows of C (0: N)
    void* c0;
    void* c1;
    const void* r;          // TE_RESID / TE_DRESID: residual rows; TE_DGELU: Gp
    const float* bias;      // [G][N]
    const float* inv_scale; // [G] or null (1)
    // TE_DGELU: column sums of C0 over each 32-row block of a tile,
    // [G][train_colpart_rows(g)][N] (tensor-core path; the SIMT path writes the
    // finished sums instead, see launch_train_gemm_simt)
    float* colpart;
    int* err;
    unsigned long long timeout_ns;
    int um_bs = 0, um_B = 0;    // TE_F16T: block size, samples
    long long um_L = 0;         // TE_F16T: values per sample
};

// Rows of C summed into one TE_DGELU partial on the tensor-core path.
constexpr int kTrainColpartRows = 32;

// Partial rows per group that the tensor-core path writes for g: whole tiles
// of 128 rows (one CTA) or 256 rows (a CTA pair) in 32-row blocks; never more
// than ceil(m_valid / 256) * 8.
int train_colpart_rows(const TrainGemm& g, int num_sms);

// tcgen05 path: fp16 operands (A and B), N a multiple of 256, K-major inner
// extents multiples of 64, MN-major inner extents multiples of 128 (A) / 256 (B).
bool train_tc_supported(const TrainGemm& g);
cudaError_t launch_train_gemm_tc(int epi, const TrainGemm& g, int num_sms, cudaStream_t s);

// SIMT path for any shape: operands and aux values are float for F32 contexts
// and fp16 for BF16 contexts.  TE_DGELU writes the finished column sums (over
// all m_valid rows, unscaled) into colpart [G][N].
cudaError_t launch_train_gemm_simt(Act act, int epi, const TrainGemm& g, cudaStream_t s);

// ---- row kernels ---------------------------------------------------------------
// S[t][b][:] = LN1(Mix(X[b])[t] + X[b][t]) in the operand type (fp16 for BF16
// contexts), with the normalised row yhat (fp16, or float for F32 contexts)
// in Yh [T][Bcap][D] and 1 / sqrt(var + eps) in rstd [T][Bcap].  X is
// sample-major in the caller dtype, or float when x_f32.
cudaError_t launch_ln1_recompute(Act act, bool x_f32, const void* X, void* S, void* Yh, float* rstd, const float* g1,
                                 const float* be1, int B, int T, int D, int Bcap, float eps, int num_sms,
                                 cudaStream_t s);

// LN2 backward.  Z [T][Bcap][D] (aux type), G sample-major [B][T][D] float:
// dZ = LN2 backward of G (float, token-major); per (token, CTA) partial sums
// [T][nblk][D] of dZ, G * zhat and G, and the largest |dZ| of each (token,
// CTA) in part_max [T][nblk], nblk = ln2_bwd_blocks(act, B, T, D, num_sms)
// (never above its value at max_batch).  Bulk-copy waits are bounded
// (timeout_ns, error word err).
int ln2_bwd_blocks(Act act, int B, int T, int D, int num_sms);
cudaError_t launch_ln2_backward(Act act, const void* Z, const float* G, const float* g2, float* dZ, float* part_db2,
                                float* part_dg2, float* part_dbe2, float* part_max, int B, int T, int D, int Bcap,
                                float eps, int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s);

// Per-token scale of the gradient operands: s_t = 2^(9 - e) with 2^e >= the
// largest |dZ| of token t (1 when it is 0); inv_scale[t] = 1 / s_t and
// dZh[t][b][:] = fp16(s_t dZ[t][b][:]) for b < B.
cudaError_t launch_grad_scale(const float* dZ, const float* part_max, int nblk, float* inv_scale, void* dZh, int B,
                              int T, int D, int Bcap, cudaStream_t s);

// LN1 and mixing backward from the recompute's yhat and rstd: dS [T][Bcap][D]
// float, dX = dY + P^T dY sample-major float with dY the LN1 backward of dS.
// Per-CTA partial sums [grid][D] of dS * yhat and dS, grid from ln1_bwd_grid
// (which never exceeds ln1_bwd_grid(max_batch, T, D, num_sms)).
// When the sample's dS rows fit in shared memory the kernel stages them with
// bulk copies; its wait on them is bounded (timeout_ns, error word err).
int ln1_bwd_grid(int B, int T, int D, int num_sms);
cudaError_t launch_ln1_mix_backward(Act act, const void* Yh, const float* rstd, const float* dS, const float* g1,
                                    float* dX, float* part_dg1, float* part_dbe1, int B, int T, int D, int Bcap,
                                    int grid, int* err, unsigned long long timeout_ns, cudaStream_t s);

// out[g][n] = sum over r < R of in[g][r][n] (fixed order), and, when
// out_all is not null, out_all[n] = sum over g of out[g][n].
cudaError_t launch_sum_rows(const float* in, float* out, float* out_all, int G, int R, int N, cudaStream_t s);

// out[i] = fp16(in[i]) for n bf16 values (saturating at +-65504).
cudaError_t launch_bf16_to_f16(const void* in, void* out, long long n, cudaStream_t s);

// G[b][t][:] = dpooled[b][:] / T  (the mean pool's backward).
cudaError_t launch_pool_backward(const float* dpooled, float* G, int B, int T, int D, cudaStream_t s);

// Prediction head: p[i] = sigmoid(pooled[i] . w + b); with labels y also the
// per-sample loss and dO[i] = gscale (p[i] - y[i]) w (any output may be null).
cudaError_t launch_head(const float* pooled, const float* w, float b, const float* y, float* p, float* loss, float* dO,
                        float gscale, int B, int D, cudaStream_t s);

// Tokenization backward helpers.  For a sample-major gradient G [B][T][D]:
// the per-token power-of-two scale (part: [T][nparts] scratch) with
// Gh = fp16(s_t G) and inv_scale[t] = 1 / s_t; and db[t][k] = sum_b G[b][t][k].
cudaError_t launch_token_grad_scale(const float* G, float* part, int nparts, float* inv_scale, void* Gh, int B, int T,
                                    int D, cudaStream_t s);
cudaError_t launch_token_colsum(const float* G, float* db, int B, int T, int D, cudaStream_t s);

// Test hook: out[2i] = Gelu(u[i]), out[2i+1] = Gelu'(u[i]) as the backward epilogues compute them.
cudaError_t launch_debug_gelu_grad(const float* u, float* out, long long n, cudaStream_t s);

}  // namespace rm
