// Internal interface of the Sparse-MoE per-token FFN ("RankMixer: Scaling Up
// Ranking Models in Industrial Recommenders", section 3.4 Eq. 10, inference
// router h_infer): per token t, E experts of their own, gates
// G = ReLU(s Wg_t + bg_t), v = sum_e G_e FFN_{t,e}(s); experts with G = 0 are
// skipped.
#pragma once

#include <cuda_runtime.h>

#include <functional>

#include "rm_internal.h"

namespace rm {

constexpr int kMoeMaxExperts = 64;

struct MoeShape {
    Act act;
    int T, D, E, Fe;
};

// Packed, device-resident expert parameters of one layer.
struct MoeWeights {
    void* W1p = nullptr;   // [T*E][Fe][D]   expert layer 1, K-major, operand type
    void* W2p = nullptr;   // [T*E][D][Fe]   expert layer 2, K-major, operand type
    float* b1 = nullptr;   // [T*E][Fe]
    float* b2 = nullptr;   // [T*E][D]
    float* Wg = nullptr;   // [T][E][D]      router, transposed, fp32
    float* bg = nullptr;   // [T][E]
};

// Workspace sized for Bcap samples (worst case: every expert active for every sample).
struct MoeWorkspace {
    int Bcap = 0;
    float* gates = nullptr;     // [B][T][E]
    int* counts = nullptr;      // [T*E] open samples per group g = t*E + e
    int* offsets = nullptr;     // [T*E + 1] first packed row of each group: g * Bcap
    float* row_gate = nullptr;  // [T*E][Bcap] gate of each packed row (first counts[g] used)
    int* slot_of = nullptr;     // [Bcap][T][E] packed row of (b, t, e) inside group t*E + e, -1 when closed
    int* tile_prefix = nullptr; // [T*E + 1] exclusive prefix of 128-row tiles over the groups
    int* tile_prefix256 = nullptr; // [T*E + 1] the same over 256-row tiles
    void* Sg = nullptr;         // [T*E*Bcap][D]  gathered LN1 rows (operand type); after expert
                                //                 layer 1 it holds the gated expert outputs Y
    void* Hm = nullptr;         // [T*E*Bcap][Fe] expert hidden activations (operand type)
};

struct MoeLaunch {
    Act act;
    const void* S;
    bool S_sample_major;       // S is the caller's [B][T][D] (caller dtype) or the stack's
                               // token-major [T][Bcap][D] (operand type)
    int T, D, E, Fe, B, Bcap, num_sms;
    int* err;                  // device error word for bounded waits (nullable)
};

cudaError_t moe_pack_weights(const MoeShape& ms, const void* Wg, const void* bg, const void* eW1, const void* eb1,
                             const void* eW2, const void* eb2, MoeWeights& w, long long* bytes, cudaStream_t s);
void moe_free_weights(MoeWeights& w);
cudaError_t moe_alloc_workspace(const MoeShape& ms, int Bcap, MoeWorkspace& ws, long long* bytes);
void moe_free_workspace(MoeWorkspace& ws);

// V[b,t] = sum_e G[b,t,e] FFN_{t,e}(S[b,t]).  V is float32, token-major
// ([T][Bcap][D]) or sample-major ([B][T][D]); gates_out (nullable) receives G
// as [B][T][E].  prof_begin(kind)/prof_end(handle) bracket each launch.
cudaError_t moe_forward(const MoeLaunch& ml, const MoeWeights& w, MoeWorkspace& ws, float* V, bool V_token_major,
                        float* gates_out, cudaStream_t s, const std::function<void*(int)>& prof_begin,
                        const std::function<void(void*)>& prof_end);

// A router alone ([T][D][E] in the caller dtype, bias [T][E]) packed as the
// expert weights' router is: float32, transposed to [T][E][D].
cudaError_t moe_pack_router(const MoeShape& ms, const void* Wg, const void* bg, float** Wg_out, float** bg_out,
                            long long* bytes, cudaStream_t s);

// G[b][t][e] = ReLU(S[b][t] . Wg[t][e] + bg[t][e]) for a packed router; S is
// sample-major [B][T][D] in the caller dtype.
cudaError_t moe_router_gates(Act act, const void* S, const float* Wg, const float* bg, float* G, int B, int T,
                             int D, int E, cudaStream_t s);

// lreg[b] = sum over t, e of G[b][t][e] and A[e] = sum over b, t of G[b][t][e]
// (either may be null), in a fixed order.
cudaError_t moe_gate_sums(const float* G, float* lreg, float* A, int B, int T, int E, cudaStream_t s);

// Z[t][b][:] = V[t][b][:] + S[t][b][:]; token-major, V float32, S and Z in the operand type.
cudaError_t moe_residual_z(Act act, const float* V, const void* S, void* Z, int B, int T, int D, int Bcap,
                           cudaStream_t s);

}  // namespace rm
