// Internal launchers of UniMixing ("UniMixer: A Unified Architecture for
// Scaling Laws in Recommendation Systems", section 4.3 Eq. 11-15), the
// learned block-Kronecker mixing that replaces TokenMixing in a layer.
// Not part of the public ABI.
//
// Per sample, flatten(X) (L = T D values) is cut into nb = L / bs blocks x_j of
// bs values.  The local step is h_j = x_j WB_j (WB_j bs x bs); the global step
// is out_i = sum_j WG[i][j] h_j (WG nb x nb).  On the device the local outputs
// of all samples are laid out as one matrix H [nb][Npitch] with column
// b * bs + r holding h_j[r] of sample b, so that the global step is a single
// dense product WG H (M = nb, N = B bs, K = nb) on the tensor cores, whose
// epilogue stores element (i, b bs + r) at Y[b][i bs + r] (sample-major).
#pragma once

#include <cuda_runtime.h>

#include "rm_internal.h"

namespace rm {

// Constrained weights (Eq. 15) of `count` n x n matrices W (float32):
// C = (W + W^T) / (2 tau); P = Sinkhorn-Knopp(exp(C)) after `iters` rounds,
// each a row then a column normalisation.  Computed in the log domain as
// P[i][j] = exp(C[i][j] + f[i] + g[j]) with f[i] = -LSE_j(C[i][j] + g[j]) and
// g[j] = -LSE_i(C[i][j] + f[i]) (the same values as the alternating
// normalisation, without overflow for small tau).  Scratch: C (count n n),
// f and g (count n each).  P32 receives P in float32; P16, when not null, a
// fp16 copy.
cudaError_t launch_sinkhorn(const float* W, int count, int n, float tau, int iters, float* C, float* f, float* g,
                            float* P32, void* P16, cudaStream_t s);

// Local step: H[j][b bs + r] = sum_s x_b[j bs + s] WB[j][s][r] for b < B,
// and 0 for the padding columns B bs <= n < Npad of every row.  X holds B
// samples of L = nb bs values, `x_stride` apart, in type xt (caller dtype or
// the operand type); H is the operand type of act (fp16 for bf16 contexts).
// bf16 contexts with bs in {16, 32, 48, 64} run it on the tensor cores
// (mma.sync, fp16 operands) from the transposed fp16 copy WBt16 [nb][bs][bs]
// (row r, column s = WB[j][s][r], see launch_unimix_pack_wb), otherwise on the
// CUDA cores from WB (float32).  The tensor-core step stages X through shared
// memory when X and H are 16-byte aligned (bounded waits: a stalled copy
// latches kDevErrTimeout in *err after timeout_ns and the kernel returns).
enum class XType { BF16, F16, F32 };
cudaError_t launch_unimix_local(XType xt, Act act, const void* X, long long x_stride, const float* WB,
                                const void* WBt16, void* H, int B, int nb, int bs, long long Npitch, long long Npad,
                                int num_sms, int* err, unsigned long long timeout_ns, cudaStream_t s);
bool unimix_local_mma_ok(int bs);
cudaError_t launch_unimix_pack_wb(const float* WB, void* WBt16, int nb, int bs, cudaStream_t s);

// Residual + LN1 after the global step: S[t][b][:] = LN1(X[b][t][:] + Y[b][t][:])
// in the operand type (token-major [T][Bcap][D]); Y is the global product,
// sample-major [B][T D] in the operand type.
cudaError_t launch_unimix_ln1(XType xt, Act act, const void* X, const void* Y, void* S, const float* g1,
                              const float* be1, int B, int T, int D, int Bcap, float eps, int num_sms,
                              cudaStream_t s);

// out[i] = Y[i] in the caller dtype, or float32 when out_f32 (n values).
cudaError_t launch_unimix_out(Act act, const void* Y, void* out, bool out_f32, long long n, cudaStream_t s);

// X_out[b][t][:] = LN2(Z[t][b][:]) in the operand type (fp16 for bf16
// contexts): a UniMixing layer's input when it follows another layer.  stats:
// nchunk (mean, M2) partials of cw columns per row (nchunk = 1: merged rows).
cudaError_t launch_ln2_out_op(Act act, const void* Z, const float2* stats, int nchunk, int cw, const float* g2,
                              const float* be2, void* X_out, int B, int T, int D, int Bcap, float eps, int num_sms,
                              cudaStream_t s);

}  // namespace rm
