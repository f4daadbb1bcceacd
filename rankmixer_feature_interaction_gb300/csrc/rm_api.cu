// C-ABI of librankmixer.so: context creation (validation, weight packing,
// workspace), the block / stack / MoE entry points, error reporting and the
// per-kernel event timer.  Declared in include/rankmixer.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/rankmixer.h"
#include "rm_internal.h"
#include "rm_moe.h"
#include "rm_train.h"
#include "rm_unimix.h"

using namespace rm;

namespace {
struct AllocBook;
AllocBook& book();
void read_fault_env(AllocBook& b);
bool alloc_failure_was_injected();
}  // namespace

namespace {

thread_local std::string g_last_error;

rm_status fail(rm_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

// The condition text of the last failed launcher check of the debug build
// (thread-local: set and read within one API call on one thread).
thread_local const char* t_bounds_what = nullptr;

}  // namespace

cudaError_t rm::debug_bounds_fail(const char* what) {
    t_bounds_what = what;
    return cudaErrorInvalidValue;
}

namespace {

rm_status cuda_fail(cudaError_t e, const char* what) {
    if (e == cudaErrorInvalidValue && t_bounds_what) {
        const char* cond = t_bounds_what;
        t_bounds_what = nullptr;
        return fail(RM_ERR_INVALID_ARG, "%s: bounds check failed: %s", what, cond);
    }
    if (e == cudaErrorMemoryAllocation)
        return fail(RM_ERR_OOM, "%s: %s", what,
                    alloc_failure_was_injected() ? "injected failure (device allocation)" : cudaGetErrorString(e));
    if (e == cudaErrorNotSupported) return fail(RM_ERR_UNSUPPORTED, "%s: shape not supported by this kernel", what);
    return fail(RM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define RM_CHECK_CUDA(expr, what)                  \
    do {                                           \
        cudaError_t _e = (expr);                   \
        if (_e != cudaSuccess) return cuda_fail(_e, what); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Default bound of every device-side wait (2 s of global time).
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;
// Up to this batch the dense PFFN leaves its LN2 row statistics as the GEMM2
// chunk partials and the consumers merge them (no separate merge launch).
constexpr int kMergeInConsumerMaxB = 256;
// Pipelined host entry: batches of at least 2 kHostChunkMin samples run as
// chunks (at most kHostChunksMax; the schedule is in rm_stack_forward_host).
constexpr int kHostChunksMax = 4;
constexpr int kHostChunkMin = 1024;

// ---- device allocations: bookkeeping and injected failures ------------------------
struct AllocBook {
    std::mutex mu;
    std::unordered_map<void*, size_t> live;
    long long made = 0;        // successful allocations since load
    long long live_bytes = 0;
    long long fail_after = -1; // >= 0: that many more allocations succeed, then one fails
    bool env_read = false;
    bool last_injected = false;
};
AllocBook& book() {
    static AllocBook b;
    return b;
}

// RM_FAULT_INJECT=alloc:N arms the injection once, at the first allocation.
void read_fault_env(AllocBook& b) {
    if (b.env_read) return;
    b.env_read = true;
    const char* v = getenv("RM_FAULT_INJECT");
    if (v && strncmp(v, "alloc:", 6) == 0) {
        char* end = nullptr;
        const long long n = strtoll(v + 6, &end, 10);
        if (end != v + 6 && n >= 0) b.fail_after = n;
    }
}

// Whether the last failed device allocation was an injected one (read once).
bool alloc_failure_was_injected() {
    std::lock_guard<std::mutex> lk(book().mu);
    const bool r = book().last_injected;
    book().last_injected = false;
    return r;
}

struct LayerW {
    void* W1p = nullptr;   // [T][F][D]  (K-major for GEMM1)
    void* W2p = nullptr;   // [T][D][F]  (K-major for GEMM2)
    float* b1 = nullptr;   // [T][F]
    float* b2 = nullptr;   // [T][D]
    float* g1 = nullptr;
    float* be1 = nullptr;
    float* g2 = nullptr;
    float* be2 = nullptr;
    MoeWeights moe;
    // training contexts: the dense weights again, in the pages' layout, as fp16
    // (bf16 contexts) or float, for the backward products
    void* W1t = nullptr;   // [T][D][F]
    void* W2t = nullptr;   // [T][F][D]
    // the training router of a dense-training / sparse-inference MoE layer
    float* Wg_train = nullptr;   // [T][E][D]
    float* bg_train = nullptr;   // [T][E]
    // UniMixing in place of TokenMixing (set by rm_set_unimixing; um_bs = 0:
    // TokenMixing): the constrained weights, WG [nb][nb] in float32 and in the
    // operand type of the global product, WB [nb][bs][bs] in float32
    int um_bs = 0;
    float* umWG32 = nullptr;
    void* umWGop = nullptr;      // fp16 (bf16 contexts); aliases umWG32 in float32 contexts
    float* umWB = nullptr;
    void* umWBt16 = nullptr;     // bf16 contexts: WB transposed ([j][r][s]) in fp16, the tensor-core
                                 // local step's B operand
};

// Activations one layer's backward reads (token-major [T][Bcap][W]): the
// LN1 output and its normalised input, the FFN's Gelu(U) and Gelu'(U), and
// the pre-LN2 rows.
struct TrainSlot {
    void* S = nullptr;        // LN1 output, operand type                 [T][Bcap][D]
    void* Yh = nullptr;       // normalised LN1 input yhat, fp16 / float  [T][Bcap][D]
    float* rstd1 = nullptr;   // LN1 1 / sqrt(var + eps) per row          [T][Bcap]
    void* A = nullptr;        // Gelu(U), operand type                    [T][Bcap][F]
    void* Gp = nullptr;       // Gelu'(U); overwritten by s_t dU          [T][Bcap][F]
    void* Z = nullptr;        // FFN output + S (pre-LN2)                 [T][Bcap][D]
};

// Workspace of the backward pass, allocated at the first training call for
// max_batch samples: slot 0 for rm_block_backward, one slot per layer for
// the stack's training forward, and the buffers every layer's backward shares.
struct TrainWS {
    bool ready = false;
    std::vector<TrainSlot> slots;
    float* dZ32 = nullptr;    // LN2 input gradient                       [T][Bcap][D]
    void* dZ = nullptr;       // s_t dZ in fp16 (bf16 contexts)           [T][Bcap][D]
    float* dS = nullptr;      // gradient at the LN1 output               [T][Bcap][D]
    float* pmax = nullptr;    // largest |dZ| per (token, row block)      [T][nblk2]
    float* inv_scale = nullptr;   // 1 / s_t                              [T]
    float* part2 = nullptr;   // LN2 partials: db2, dgamma2, dbeta2       3 x [T][nblk2][D]
    float* tmpTD = nullptr;   // per-token sums before the sum over tokens [T][D]
    float* colpart = nullptr; // db1 partials                             [T][rows][F]
    float* part1 = nullptr;   // LN1 partials: dgamma1, dbeta1            2 x [grid1][D]
    // the stack: the next layer's input (float32), the two gradient buffers, pooled scratch
    float* Xn = nullptr;      // [Bcap][T][D]
    float* G0 = nullptr;      // [Bcap][T][D]
    float* G1 = nullptr;
    float* pooled = nullptr;  // [Bcap][D]
    int nblk2 = 0, colrows = 0, grid1 = 0;
    int saved_B = 0;          // batch of the activations rm_stack_forward_train left in the slots (0: none)
};

struct Event {
    cudaEvent_t a, b;
};

}  // namespace

struct rm_ctx {
    rm_config cfg{};
    int device = 0;
    int num_sms = 0;
    Act act = Act::BF16;
    size_t esz = 2;
    int F = 0;           // kD
    bool use_tc = false;
    int nchunk = 1, cw = 0;
    std::vector<LayerW> layers;
    // workspace (token-major)
    int Bcap = 0;
    void* S = nullptr;           // operand type (fp16 for bf16 contexts)
    void* Hid = nullptr;         // operand type
    void* Z = nullptr;           // pre-LN2 rows, operand type
    float2* stats = nullptr;     // GEMM2 epilogue partials: [T][Bcap][nchunk] (mean, M2) per column chunk
    // row-block counters of the fused layer GEMM ([T][ceil(Bcap / 256)], only grow) and its launch count
    unsigned* dep_cnt = nullptr;
    unsigned dep_epoch = 0;
    float2* rows = nullptr;      // merged: [T][Bcap] (mean, M2) of each full pre-LN2 row
    // where the last PFFN left its LN2 row statistics for the consumers: the
    // merged rows, or (small batches) the GEMM2 chunk partials themselves
    const float2* ln2_st = nullptr;
    int ln2_nchunk = 1, ln2_cw = 0;
    float* V = nullptr;          // MoE PFFN output inside the stack
    MoeWorkspace moe_ws;
    TrainWS tw;
    // feature tokenization ("RankMixer" Eq. 2), set by rm_set_tokenizer
    int tok_d = 0;
    void* Wtok = nullptr;        // [T][d][D], fp16 (bf16 contexts) or float
    float* btok = nullptr;       // [T][D]
    void* Etok = nullptr;        // fp16 copy of the embeddings [Bcap][T d] (bf16 contexts)
    void* X0ws = nullptr;        // tokens for rm_score [Bcap][T][D], context dtype
    float* pooled_ws = nullptr;  // [Bcap][D]
    float* ginfer = nullptr;     // inference-router gates of the MoE training forward [Bcap][T][E]
    void* dX0h = nullptr;        // tokenization backward: s_t dX0 in fp16 [Bcap][T][D] (bf16 contexts)
    float* tok_part = nullptr;   // [T][kTokParts] per-token maxima
    float* tok_inv = nullptr;    // [T] 1 / s_t
    // UniMixing workspace: the local outputs H and the global product Yt
    // ([nb][Npitch] each, operand type, Npitch = Bcap bs rounded up to 256),
    // and a layer input after LN2 ([Bcap][T][D], operand type)
    void* umH = nullptr;
    void* umYt = nullptr;
    void* umX = nullptr;
    size_t um_bytes = 0;         // bytes of umH (and of umYt)
    // host-entry staging: device copies of X0 and pooled, the copy streams and
    // per-chunk events of the pipelined host entry
    void* X0_dev = nullptr;
    float* pooled_dev = nullptr;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[kHostChunksMax] = {}, ev_done[kHostChunksMax] = {};
    // pipelined host entry (rm_stack_forward_host_async): two device staging
    // slots, each with its copy-in, compute and copy-out events, and the ticket
    // that holds it (-1: free)
    void* hx_dev[2] = {};
    float* hp_dev[2] = {};
    cudaEvent_t hx_in[2] = {}, hx_done[2] = {}, hx_out[2] = {};
    long long h_next = 0;
    long long h_slot[2] = {-1, -1};
    // error word and the debug flag nothing sets
    int* d_err = nullptr;
    int* d_flag = nullptr;
    long long weight_bytes = 0, ws_bytes = 0;
    // profiling
    bool prof = false;
    std::vector<Event> ev_pool;
    std::vector<std::pair<int, int>> ev_used;   // (kind, pool index)
    std::vector<cudaEvent_t> spare;
};

namespace {

rm_status dmalloc(rm_ctx* c, void** p, size_t bytes, long long* counter) {
    *p = nullptr;
    if (bytes == 0) return RM_OK;
    cudaError_t e = device_alloc(p, bytes);
    if (e != cudaSuccess) {
        *p = nullptr;
        cudaGetLastError();
        return fail(RM_ERR_OOM, "device allocation of %zu bytes failed: %s", bytes,
                    e == cudaErrorMemoryAllocation && alloc_failure_was_injected() ? "injected failure"
                                                                                    : cudaGetErrorString(e));
    }
    if (counter) *counter += (long long)bytes;
    (void)c;
    return RM_OK;
}

rm_status cuda_fail(cudaError_t e, const char* what);

// The host entries' two copy streams and per-chunk events (created at first use).
rm_status copy_streams(rm_ctx* c) {
    if (c->s_in) return RM_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&c->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->s_out, cudaStreamNonBlocking);
    for (int i = 0; e == cudaSuccess && i < kHostChunksMax; ++i) {
        e = cudaEventCreateWithFlags(&c->ev_in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_done[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        // leave nothing half made: the next call starts again
        if (c->s_in) cudaStreamDestroy(c->s_in);
        if (c->s_out) cudaStreamDestroy(c->s_out);
        c->s_in = c->s_out = nullptr;
        for (int i = 0; i < kHostChunksMax; ++i) {
            if (c->ev_in[i]) cudaEventDestroy(c->ev_in[i]);
            if (c->ev_done[i]) cudaEventDestroy(c->ev_done[i]);
            c->ev_in[i] = c->ev_done[i] = nullptr;
        }
        return cuda_fail(e, "copy streams");
    }
    return RM_OK;
}

// dmalloc for a lazily allocated buffer: keeps one that an earlier call
// already allocated (a call that failed part way through a group of buffers
// leaves the ones it got; the next call completes the group).
rm_status ensure(rm_ctx* c, void** p, size_t bytes, long long* counter) {
    if (*p) return RM_OK;
    return dmalloc(c, p, bytes, counter);
}

void free_ctx(rm_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    cudaDeviceSynchronize();
    for (auto& l : c->layers) {
        device_free(l.W1p); device_free(l.W2p); device_free(l.b1); device_free(l.b2);
        device_free(l.g1); device_free(l.be1); device_free(l.g2); device_free(l.be2);
        moe_free_weights(l.moe);
        device_free(l.W1t); device_free(l.W2t); device_free(l.Wg_train); device_free(l.bg_train);
        if (l.umWGop != l.umWG32) device_free(l.umWGop);
        device_free(l.umWG32); device_free(l.umWB); device_free(l.umWBt16);
    }
    device_free(c->umH); device_free(c->umYt); device_free(c->umX);
    {
        TrainWS& t = c->tw;
        for (auto& sl : t.slots) {
            device_free(sl.S); device_free(sl.Yh); device_free(sl.rstd1); device_free(sl.A); device_free(sl.Gp); device_free(sl.Z);
        }
        device_free(t.dZ32); device_free(t.dZ); device_free(t.dS); device_free(t.pmax); device_free(t.inv_scale);
        device_free(t.part2); device_free(t.tmpTD); device_free(t.colpart); device_free(t.part1);
        device_free(t.Xn); device_free(t.G0); device_free(t.G1); device_free(t.pooled);
    }
    device_free(c->Wtok); device_free(c->btok); device_free(c->Etok); device_free(c->X0ws); device_free(c->pooled_ws);
    device_free(c->ginfer); device_free(c->dX0h); device_free(c->tok_part); device_free(c->tok_inv);
    moe_free_workspace(c->moe_ws);
    device_free(c->S); device_free(c->Hid); device_free(c->Z); device_free(c->stats); device_free(c->rows); device_free(c->V);
    device_free(c->dep_cnt);
    device_free(c->X0_dev); device_free(c->pooled_dev);
    for (int i = 0; i < kHostChunksMax; ++i) {
        if (c->ev_in[i]) cudaEventDestroy(c->ev_in[i]);
        if (c->ev_done[i]) cudaEventDestroy(c->ev_done[i]);
    }
    for (int k = 0; k < 2; ++k) {
        device_free(c->hx_dev[k]);
        device_free(c->hp_dev[k]);
        if (c->hx_in[k]) cudaEventDestroy(c->hx_in[k]);
        if (c->hx_done[k]) cudaEventDestroy(c->hx_done[k]);
        if (c->hx_out[k]) cudaEventDestroy(c->hx_out[k]);
    }
    if (c->s_in) cudaStreamDestroy(c->s_in);
    if (c->s_out) cudaStreamDestroy(c->s_out);
    device_free(c->d_err); device_free(c->d_flag);
    for (auto& e : c->ev_pool) { cudaEventDestroy(e.a); cudaEventDestroy(e.b); }
    delete c;
}

// ---- profiling --------------------------------------------------------------
// NVTX ranges around each kernel class's launches (host timeline, for nsys and
// similar tools), when RM_NVTX=1 is in the environment; names as in rm_kernel_kind.
const char* const kKindNames[RM_K_COUNT] = {
    "rm:mix_ln1", "rm:gemm1", "rm:gemm2", "rm:ln2_out", "rm:pool", "rm:rowstats", "rm:moe_route", "rm:moe_gemm1",
    "rm:moe_gemm2", "rm:misc", "rm:moe_combine", "rm:bwd_recompute", "rm:bwd_dgrad", "rm:bwd_wgrad",
    "rm:bwd_rows", "rm:tokenize", "rm:head", "rm:unimix", "rm:pffn"};

bool nvtx_on() {
    static int env = -1;
    if (env < 0) {
        const char* v = getenv("RM_NVTX");
        env = (v && v[0] == '1') ? 1 : 0;
    }
    return env == 1;
}

struct ProfScope {
    rm_ctx* c;
    int kind;
    cudaStream_t s;
    int idx = -1;
    bool nvtx = false;
    ProfScope(rm_ctx* c_, int kind_, cudaStream_t s_) : c(c_), kind(kind_), s(s_) {
        if (nvtx_on() && kind >= 0 && kind < RM_K_COUNT) {
            nvtxRangePushA(kKindNames[kind]);
            nvtx = true;
        }
        if (!c->prof) return;
        if (c->ev_used.size() >= c->ev_pool.size()) {
            Event e;
            if (cudaEventCreate(&e.a) != cudaSuccess || cudaEventCreate(&e.b) != cudaSuccess) return;
            c->ev_pool.push_back(e);
        }
        idx = (int)c->ev_used.size();
        c->ev_used.push_back({kind, idx});
        cudaEventRecord(c->ev_pool[idx].a, s);
    }
    ~ProfScope() {
        if (idx >= 0) cudaEventRecord(c->ev_pool[idx].b, s);
        if (nvtx) nvtxRangePop();
    }
};

rm_status validate_cfg(const rm_config* cfg) {
    if (!cfg) return fail(RM_ERR_INVALID_ARG, "cfg is NULL");
    if (cfg->T < 1 || cfg->D < 1 || cfg->H < 1 || cfg->k < 1 || cfg->L < 1 || cfg->max_batch < 1)
        return fail(RM_ERR_INVALID_ARG, "T, D, H, k, L and max_batch must be positive");
    if (cfg->D % cfg->H != 0) return fail(RM_ERR_INVALID_ARG, "D (%d) must be divisible by H (%d)", cfg->D, cfg->H);
    if (cfg->H != cfg->T)
        return fail(RM_ERR_UNSUPPORTED, "H (%d) must equal T (%d): the mixing residual needs a [T][D] result",
                    cfg->H, cfg->T);
    if (cfg->dtype != RM_F32 && cfg->dtype != RM_BF16) return fail(RM_ERR_INVALID_ARG, "unknown dtype");
    if (!(cfg->ln_eps >= 0.f) || !std::isfinite(cfg->ln_eps)) return fail(RM_ERR_INVALID_ARG, "ln_eps must be >= 0");
    if (cfg->L > 32) return fail(RM_ERR_UNSUPPORTED, "at most 32 layers");
    if (cfg->T > 128) return fail(RM_ERR_UNSUPPORTED, "at most 128 tokens");
    const int q = cfg->D / cfg->H;
    const bool vec2 = (q % 2 == 0) && (cfg->D % 64 == 0);
    if ((vec2 && cfg->D > 3072) || (!vec2 && cfg->D > 1536))
        return fail(RM_ERR_UNSUPPORTED, "D too large for the mixing kernel");
    if (cfg->gemm_path != RM_PATH_AUTO && cfg->gemm_path != RM_PATH_SIMT && cfg->gemm_path != RM_PATH_TCGEN05)
        return fail(RM_ERR_INVALID_ARG, "unknown gemm_path");
    if (cfg->n_experts < 0 || (cfg->n_experts > 0 && cfg->expert_hidden < 1))
        return fail(RM_ERR_INVALID_ARG, "n_experts > 0 needs expert_hidden >= 1");
    if (cfg->n_experts == 0 && cfg->moe_layer_mask != 0)
        return fail(RM_ERR_INVALID_ARG, "moe_layer_mask set without experts");
    if (cfg->n_experts > kMoeMaxExperts) return fail(RM_ERR_UNSUPPORTED, "at most %d experts", kMoeMaxExperts);
    return RM_OK;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

rm_status check_ctx(const rm_ctx* c) {
    if (!c) return fail(RM_ERR_INVALID_ARG, "ctx is NULL");
    return RM_OK;
}

rm_status check_batch(const rm_ctx* c, int B) {
    if (B < 1 || B > c->Bcap) return fail(RM_ERR_INVALID_ARG, "B (%d) must be in [1, max_batch=%d]", B, c->Bcap);
    return RM_OK;
}

// Activation outputs come in the context dtype or in float32 (the values
// before their rounding to bf16 in a bf16 context).
rm_status check_out_dtype(const rm_ctx* c, rm_dtype d, bool* out_f32) {
    if (d != RM_F32 && d != RM_BF16) return fail(RM_ERR_INVALID_ARG, "unknown output dtype %d", (int)d);
    if (d == RM_BF16 && c->act == Act::F32)
        return fail(RM_ERR_INVALID_ARG, "a float32 context writes float32 outputs (out_dtype RM_F32)");
    *out_f32 = d == RM_F32;
    return RM_OK;
}

// ---- the block steps ---------------------------------------------------------
rm_status run_pffn(rm_ctx* c, int layer, int B, cudaStream_t s) {
    const LayerW& w = c->layers[layer];
    const rm_config& g = c->cfg;
    if (g.moe_layer_mask & (1u << layer)) {
        // Sparse-MoE PFFN: V = sum_e gate * expert(S), then Z = V + S and row statistics.
        rm_status st = RM_OK;
        {
            MoeLaunch ml{c->act, c->S, /*S sample-major*/ false, g.T, g.D, g.n_experts, g.expert_hidden, B,
                         c->Bcap, c->num_sms, c->d_err};
            cudaError_t e = moe_forward(ml, w.moe, c->moe_ws, c->V, /*V token-major*/ true, nullptr, s,
                                        [&](int kind) { return (void*)new ProfScope(c, kind, s); },
                                        [](void* p) { delete (ProfScope*)p; });
            if (e != cudaSuccess) st = cuda_fail(e, "moe pffn");
        }
        if (st != RM_OK) return st;
        ProfScope ps(c, RM_K_GEMM2, s);
        RM_CHECK_CUDA(moe_residual_z(c->act, c->V, c->S, c->Z, B, g.T, g.D, c->Bcap, s), "moe residual");
        ProfScope ps2(c, RM_K_ROWSTATS, s);
        RM_CHECK_CUDA(launch_rowstats(c->act, c->Z, c->rows, B, g.T, g.D, c->Bcap, c->num_sms, s), "row stats");
        c->ln2_st = c->rows;
        c->ln2_nchunk = 1;
        c->ln2_cw = g.D;
        return RM_OK;
    }
    // Under stream capture the two launches run instead of the fused one: the
    // fused launch waits for counter values that depend on how many fused
    // launches came before (host state), which a replayed graph would not track.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    RM_CHECK_CUDA(cudaStreamIsCapturing(s, &cap), "cudaStreamIsCapturing");
    if (c->use_tc && c->dep_cnt && cap == cudaStreamCaptureStatusNone && layer_tc_fusable(B, g.D, c->F)) {
        // both GEMMs in one launch (the same bits as the two launches below)
        ProfScope ps(c, RM_K_PFFN, s);
        cudaError_t e = launch_layer_tc(c->S, w.W1p, w.b1, c->Hid, w.W2p, w.b2, c->Z, c->stats, B, g.T, g.D, c->F,
                                        c->Bcap, c->num_sms, c->dep_cnt, c->dep_epoch, c->d_err, kWaitTimeoutNs, s);
        if (e != cudaSuccess) return cuda_fail(e, (std::string("ffn layer (tcgen05) ") + tc_last_error()).c_str());
        ++c->dep_epoch;
    } else if (c->use_tc) {
        {
            ProfScope ps(c, RM_K_GEMM1, s);
            cudaError_t e = launch_gemm1_tc(c->S, w.W1p, w.b1, c->Hid, B, g.T, g.D, c->F, c->Bcap, c->num_sms,
                                            c->d_err, kWaitTimeoutNs, s);
            if (e != cudaSuccess) return cuda_fail(e, (std::string("gemm1 (tcgen05) ") + tc_last_error()).c_str());
        }
        {
            ProfScope ps(c, RM_K_GEMM2, s);
            cudaError_t e = launch_gemm2_tc(c->Hid, w.W2p, w.b2, c->S, c->Z, c->stats, B, g.T, g.D, c->F, c->Bcap,
                                            c->num_sms, c->d_err, kWaitTimeoutNs, s);
            if (e != cudaSuccess) return cuda_fail(e, (std::string("gemm2 (tcgen05) ") + tc_last_error()).c_str());
        }
    }
    if (c->use_tc) {
        if (B <= kMergeInConsumerMaxB) {
            // small batches: the consumers merge the chunk partials themselves (one
            // launch fewer; the merge costs them next to nothing at this size)
            c->ln2_st = c->stats;
            c->ln2_nchunk = c->nchunk;
            c->ln2_cw = c->cw;
            return RM_OK;
        }
        ProfScope ps(c, RM_K_ROWSTATS, s);
        RM_CHECK_CUDA(launch_stats_finalize(c->stats, c->rows, B, g.T, c->Bcap, c->nchunk, c->cw, c->num_sms, s),
                      "row statistics");
    } else {
        {
            ProfScope ps(c, RM_K_GEMM1, s);
            RM_CHECK_CUDA(launch_gemm1_simt(c->act, c->S, w.W1p, w.b1, c->Hid, B, g.T, g.D, c->F, c->Bcap, s),
                          "gemm1 (simt)");
        }
        {
            ProfScope ps(c, RM_K_GEMM2, s);
            RM_CHECK_CUDA(launch_gemm2_simt(c->act, c->Hid, w.W2p, w.b2, c->S, c->Z, B, g.T, g.D, c->F, c->Bcap, s),
                          "gemm2 (simt)");
        }
        ProfScope ps(c, RM_K_ROWSTATS, s);
        RM_CHECK_CUDA(launch_rowstats(c->act, c->Z, c->rows, B, g.T, g.D, c->Bcap, c->num_sms, s), "row stats");
    }
    c->ln2_st = c->rows;
    c->ln2_nchunk = 1;
    c->ln2_cw = g.D;
    return RM_OK;
}

MixLnArgs mix_args(const rm_ctx* c, int layer, int B) {
    MixLnArgs a{};
    const rm_config& g = c->cfg;
    a.S = c->S;
    a.g1 = c->layers[layer].g1;
    a.be1 = c->layers[layer].be1;
    a.B = B;
    a.T = g.T;
    a.D = g.D;
    a.q = g.D / g.H;
    a.Bcap = c->Bcap;
    a.eps = g.ln_eps;
    a.err = c->d_err;
    a.timeout_ns = kWaitTimeoutNs;
    return a;
}

// UniMixing layers (defined with the backward helpers below)
XType caller_xtype(const rm_ctx* c);
XType op_xtype(const rm_ctx* c);
rm_status unimix_mix_ln1(rm_ctx* c, int layer, const void* X, XType xt, int B, cudaStream_t s);

rm_status stack_device(rm_ctx* c, const void* X0, float* pooled, void* XL, bool xl_f32, int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    for (int n = 0; n < g.L; ++n) {
        MixLnArgs a = mix_args(c, n, B);
        if (c->layers[n].um_bs) {
            const void* xin = X0;
            XType xt = caller_xtype(c);
            if (n > 0) {
                ProfScope ps(c, RM_K_LN2_OUT, s);
                RM_CHECK_CUDA(launch_ln2_out_op(c->act, c->Z, c->ln2_st, c->ln2_nchunk, c->ln2_cw,
                                                c->layers[n - 1].g2, c->layers[n - 1].be2,
                                                c->umX, B, g.T, g.D, c->Bcap, g.ln_eps, c->num_sms, s),
                              "ln2 (unimixing layer input)");
                xin = c->umX;
                xt = op_xtype(c);
            }
            rm_status st = unimix_mix_ln1(c, n, xin, xt, B, s);
            if (st != RM_OK) return st;
        } else if (n == 0) {
            a.X = X0;
            ProfScope ps(c, RM_K_MIX_LN1, s);
            RM_CHECK_CUDA(launch_mix_ln1(c->act, false, a, c->num_sms, s), "mix+ln1");
        } else {
            a.Z = c->Z;
            a.stats = c->ln2_st;
            a.g2 = c->layers[n - 1].g2;
            a.be2 = c->layers[n - 1].be2;
            a.nchunk = c->ln2_nchunk;
            a.cw = c->ln2_cw;
            ProfScope ps(c, RM_K_MIX_LN1, s);
            RM_CHECK_CUDA(launch_mix_ln1(c->act, true, a, c->num_sms, s), "ln2+mix+ln1");
        }
        rm_status st = run_pffn(c, n, B, s);
        if (st != RM_OK) return st;
    }
    const int last = g.L - 1;
    ProfScope ps(c, RM_K_POOL, s);
    RM_CHECK_CUDA(launch_pool(c->act, c->Z, c->ln2_st, c->layers[last].g2, c->layers[last].be2, pooled, XL, xl_f32,
                              B, g.T, g.D, c->Bcap, c->ln2_nchunk, c->ln2_cw, g.ln_eps, c->num_sms,
                              c->d_err, kWaitTimeoutNs, s),
                  "ln2+pool");
    return RM_OK;
}

rm_status pack_layer(rm_ctx* c, const rm_layer_params& p, LayerW& w, cudaStream_t s) {
    const rm_config& g = c->cfg;
    const int T = g.T, D = g.D, F = c->F;
    if (!p.W1 || !p.b1 || !p.W2 || !p.b2 || !p.ln1_gamma || !p.ln1_beta || !p.ln2_gamma || !p.ln2_beta)
        return fail(RM_ERR_INVALID_ARG, "a dense layer parameter pointer is NULL");
    rm_status st;
    if ((st = dmalloc(c, &w.W1p, (size_t)T * F * D * c->esz, &c->weight_bytes)) != RM_OK) return st;
    if ((st = dmalloc(c, &w.W2p, (size_t)T * D * F * c->esz, &c->weight_bytes)) != RM_OK) return st;
    if ((st = dmalloc(c, (void**)&w.b1, (size_t)T * F * 4, &c->weight_bytes)) != RM_OK) return st;
    if ((st = dmalloc(c, (void**)&w.b2, (size_t)T * D * 4, &c->weight_bytes)) != RM_OK) return st;
    float** lnp[4] = {&w.g1, &w.be1, &w.g2, &w.be2};
    const void* lns[4] = {p.ln1_gamma, p.ln1_beta, p.ln2_gamma, p.ln2_beta};
    for (int i = 0; i < 4; ++i)
        if ((st = dmalloc(c, (void**)lnp[i], (size_t)D * 4, &c->weight_bytes)) != RM_OK) return st;
    // W1 [T][D][F] -> W1p [T][F][D];  W2 [T][F][D] -> W2p [T][D][F]
    RM_CHECK_CUDA(launch_pack_transpose(c->act, p.W1, w.W1p, T, D, F, s), "pack W1");
    RM_CHECK_CUDA(launch_pack_transpose(c->act, p.W2, w.W2p, T, F, D, s), "pack W2");
    RM_CHECK_CUDA(launch_to_f32(c->act, p.b1, w.b1, (size_t)T * F, s), "pack b1");
    RM_CHECK_CUDA(launch_to_f32(c->act, p.b2, w.b2, (size_t)T * D, s), "pack b2");
    for (int i = 0; i < 4; ++i) RM_CHECK_CUDA(launch_to_f32(c->act, lns[i], *lnp[i], (size_t)D, s), "pack LN");
    if (g.training) {
        // the caller's W1 [T][D][F] and W2 [T][F][D] in their layout: float as
        // they are, bf16 converted to fp16 (exact apart from |w| < 2^-14)
        const long long n = (long long)T * D * F;
        const size_t wb = (size_t)n * c->esz;
        if ((st = dmalloc(c, &w.W1t, wb, &c->weight_bytes)) != RM_OK) return st;
        if ((st = dmalloc(c, &w.W2t, wb, &c->weight_bytes)) != RM_OK) return st;
        if (c->act == Act::F32) {
            RM_CHECK_CUDA(cudaMemcpyAsync(w.W1t, p.W1, wb, cudaMemcpyDeviceToDevice, s), "copy W1");
            RM_CHECK_CUDA(cudaMemcpyAsync(w.W2t, p.W2, wb, cudaMemcpyDeviceToDevice, s), "copy W2");
        } else {
            RM_CHECK_CUDA(launch_bf16_to_f16(p.W1, w.W1t, n, s), "copy W1");
            RM_CHECK_CUDA(launch_bf16_to_f16(p.W2, w.W2t, n, s), "copy W2");
        }
    }
    if (g.n_experts > 0) {
        if (!p.Wg || !p.bg || !p.eW1 || !p.eb1 || !p.eW2 || !p.eb2)
            return fail(RM_ERR_INVALID_ARG, "a Sparse-MoE parameter pointer is NULL");
        MoeShape ms{c->act, T, D, g.n_experts, g.expert_hidden};
        cudaError_t e = moe_pack_weights(ms, p.Wg, p.bg, p.eW1, p.eb1, p.eW2, p.eb2, w.moe, &c->weight_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "pack MoE weights");
        if ((p.Wg_train == nullptr) != (p.bg_train == nullptr))
            return fail(RM_ERR_INVALID_ARG, "Wg_train and bg_train must both be set or both be NULL");
        if (p.Wg_train) {
            e = moe_pack_router(ms, p.Wg_train, p.bg_train, &w.Wg_train, &w.bg_train, &c->weight_bytes, s);
            if (e != cudaSuccess) return cuda_fail(e, "pack the training router");
        }
    }
    return RM_OK;
}

// ---- backward pass ------------------------------------------------------------------
// nslots: how many activation slots the call needs (1 for a block, L for the stack).
rm_status train_ws_ready(rm_ctx* c, int nslots, bool stack) {
    TrainWS& t = c->tw;
    const rm_config& g = c->cfg;
    const size_t T = g.T, D = g.D, F = c->F, Bc = c->Bcap;
    const size_t osz = op_size(c->act);                    // operands, yhat, Gelu'(U) and Z: fp16 or float
    rm_status st;
    if (!t.ready) {
        t.nblk2 = ln2_bwd_blocks(c->act, c->Bcap, g.T, g.D, c->num_sms);
        t.colrows = (c->Bcap + 255) / 256 * (256 / kTrainColpartRows);   // covers 128- and 256-row tiles
        t.grid1 = ln1_bwd_grid(c->Bcap, g.T, g.D, c->num_sms);
        if ((st = ensure(c, (void**)&t.dZ32, T * Bc * D * 4, &c->ws_bytes)) != RM_OK ||
            (c->act != Act::F32 && (st = ensure(c, &t.dZ, T * Bc * D * osz, &c->ws_bytes)) != RM_OK) ||
            (st = ensure(c, (void**)&t.dS, T * Bc * D * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.pmax, T * (size_t)t.nblk2 * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.inv_scale, T * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.part2, 3 * T * (size_t)t.nblk2 * D * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.tmpTD, T * D * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.colpart, T * (size_t)t.colrows * F * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.part1, 2 * (size_t)t.grid1 * D * 4, &c->ws_bytes)) != RM_OK)
            return st;
        t.ready = true;
    }
    while ((int)t.slots.size() < nslots) {
        TrainSlot sl;
        if ((st = dmalloc(c, &sl.S, T * Bc * D * osz, &c->ws_bytes)) != RM_OK ||
            (st = dmalloc(c, &sl.Yh, T * Bc * D * osz, &c->ws_bytes)) != RM_OK ||
            (st = dmalloc(c, (void**)&sl.rstd1, T * Bc * 4, &c->ws_bytes)) != RM_OK ||
            (st = dmalloc(c, &sl.A, T * Bc * F * osz, &c->ws_bytes)) != RM_OK ||
            (st = dmalloc(c, &sl.Gp, T * Bc * F * osz, &c->ws_bytes)) != RM_OK ||
            (st = dmalloc(c, &sl.Z, T * Bc * D * osz, &c->ws_bytes)) != RM_OK) {
            // a slot is used whole or not at all
            device_free(sl.S); device_free(sl.Yh); device_free(sl.rstd1); device_free(sl.A); device_free(sl.Gp);
            device_free(sl.Z);
            return st;
        }
        t.slots.push_back(sl);
    }
    if (stack) {
        if ((st = ensure(c, (void**)&t.Xn, Bc * T * D * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.G0, Bc * T * D * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.G1, Bc * T * D * 4, &c->ws_bytes)) != RM_OK ||
            (st = ensure(c, (void**)&t.pooled, Bc * D * 4, &c->ws_bytes)) != RM_OK)
            return st;
    }
    return RM_OK;
}

rm_status check_grads(const rm_layer_grads* gr) {
    if (!gr) return fail(RM_ERR_INVALID_ARG, "grads is NULL");
    const float* p[8] = {gr->dW1, gr->db1, gr->dW2, gr->db2, gr->dln1_gamma, gr->dln1_beta, gr->dln2_gamma,
                         gr->dln2_beta};
    for (const float* q : p) {
        if (!q) return fail(RM_ERR_INVALID_ARG, "a gradient buffer is NULL");
        if (!aligned16(q)) return fail(RM_ERR_INVALID_ARG, "gradient buffers must be 16-byte aligned");
    }
    return RM_OK;
}

TrainGemm train_gemm_base(rm_ctx* c) {
    TrainGemm m{};
    m.G = c->cfg.T;
    m.err = c->d_err;
    m.timeout_ns = kWaitTimeoutNs;
    return m;
}

rm_status run_train_gemm(rm_ctx* c, int epi, const TrainGemm& m, bool* used_tc, const char* what, cudaStream_t s) {
    const bool tc = c->use_tc && train_tc_supported(m);
    if (used_tc) *used_tc = tc;
    cudaError_t e = tc ? launch_train_gemm_tc(epi, m, c->num_sms, s) : launch_train_gemm_simt(c->act, epi, m, s);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return RM_OK;
}

// The forward of dense layer `layer` into activation slot `slot`, keeping
// what its backward reads: S = LN1(Mix(X) + X) with yhat and rstd,
// A = Gelu(U) and Gp = Gelu'(U) for U = S W1 + b1, and Z = A W2 + b2 + S.
// X is the layer input, sample-major, in the context dtype or (x_f32) float32.
rm_status train_layer_forward(rm_ctx* c, int layer, int slot, const void* X, bool x_f32, int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    const LayerW& w = c->layers[layer];
    TrainSlot& sl = c->tw.slots[slot];
    const int T = g.T, D = g.D, F = c->F, Bc = c->Bcap;
    const long long BcD = (long long)Bc * D, BcF = (long long)Bc * F, DF = (long long)D * F;
    ProfScope ps(c, RM_K_BWD_RECOMPUTE, s);
    RM_CHECK_CUDA(launch_ln1_recompute(c->act, x_f32, X, sl.S, sl.Yh, sl.rstd1, w.g1, w.be1, B, T, D, Bc, g.ln_eps,
                                       c->num_sms, s),
                  "ln1 (training forward)");
    rm_status st;
    TrainGemm m = train_gemm_base(c);
    m.M = B; m.N = F; m.K = D; m.m_valid = B;
    m.a = {sl.S, D, B, BcD, false};
    m.b = {w.W1t, F, D, DF, true};
    m.c_gpitch = BcF; m.c0 = sl.A; m.c1 = sl.Gp; m.bias = w.b1;
    if ((st = run_train_gemm(c, TE_GELU2, m, nullptr, "ffn layer 1 (training forward)", s)) != RM_OK) return st;
    m = train_gemm_base(c);
    m.M = B; m.N = D; m.K = F; m.m_valid = B;
    m.a = {sl.A, F, B, BcF, false};
    m.b = {w.W2t, D, F, DF, true};
    m.c_gpitch = BcD; m.c0 = sl.Z; m.r = sl.S; m.bias = w.b2;
    return run_train_gemm(c, TE_RESID, m, nullptr, "ffn layer 2 (training forward)", s);
}

// The backward of dense layer `layer` from the activations in slot `slot`
// (written by train_layer_forward for the same batch): G = dl/dX' at the
// layer output (float32 [B][T][D]) -> dX (float32 [B][T][D]) and the
// parameter gradients.  Consumes the slot's Gelu'(U) (replaced by s_t dU).
rm_status train_layer_backward(rm_ctx* c, int layer, int slot, const float* G, float* dX, const rm_layer_grads& gr,
                               int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    const LayerW& w = c->layers[layer];
    TrainWS& t = c->tw;
    TrainSlot& sl = t.slots[slot];
    const int T = g.T, D = g.D, F = c->F, Bc = c->Bcap;
    const long long BcD = (long long)Bc * D, BcF = (long long)Bc * F, DF = (long long)D * F;
    rm_status st;
    const int nblk = ln2_bwd_blocks(c->act, B, T, D, c->num_sms);
    float* p_db2 = t.part2;
    float* p_dg2 = t.part2 + (size_t)T * t.nblk2 * D;
    float* p_dbe2 = t.part2 + 2 * (size_t)T * t.nblk2 * D;
    // dZ as a GEMM operand: float for float32 contexts; s_t dZ in fp16 otherwise
    const void* dZop = t.dZ32;
    const float* inv = nullptr;
    {
        ProfScope ps(c, RM_K_BWD_ROWS, s);
        RM_CHECK_CUDA(launch_ln2_backward(c->act, sl.Z, G, w.g2, t.dZ32, p_db2, p_dg2, p_dbe2, t.pmax, B, T, D, Bc,
                                          g.ln_eps, c->num_sms, c->d_err, kWaitTimeoutNs, s),
                      "ln2 backward");
        if (c->act != Act::F32) {
            RM_CHECK_CUDA(launch_grad_scale(t.dZ32, t.pmax, nblk, t.inv_scale, t.dZ, B, T, D, Bc, s), "grad scale");
            dZop = t.dZ;
            inv = t.inv_scale;
        }
    }
    {   // dW2 = A^T dZ
        ProfScope ps(c, RM_K_BWD_WGRAD, s);
        TrainGemm m = train_gemm_base(c);
        m.M = F; m.N = D; m.K = B; m.m_valid = F;
        m.a = {sl.A, F, B, BcF, true};
        m.b = {dZop, D, B, BcD, true};
        m.c_gpitch = DF; m.c0 = gr.dW2; m.inv_scale = inv;
        if ((st = run_train_gemm(c, TE_F32, m, nullptr, "dW2", s)) != RM_OK) return st;
    }
    bool db1_partials = false;
    int colrows = 0;
    void* dU = sl.Gp;     // s_t dU = (s_t dZ W2^T) * Gelu'(U) replaces Gelu'(U) element by element
    {
        ProfScope ps(c, RM_K_BWD_DGRAD, s);
        TrainGemm m = train_gemm_base(c);
        m.M = B; m.N = F; m.K = D; m.m_valid = B;
        m.a = {dZop, D, B, BcD, false};
        m.b = {w.W2t, D, F, DF, false};
        m.c_gpitch = BcF; m.c0 = dU; m.r = sl.Gp; m.inv_scale = inv;
        const bool tc = c->use_tc && train_tc_supported(m);
        m.colpart = tc ? t.colpart : gr.db1;
        colrows = tc ? train_colpart_rows(m, c->num_sms) : 0;
        if ((st = run_train_gemm(c, TE_DGELU, m, &db1_partials, "dU", s)) != RM_OK) return st;
        m = train_gemm_base(c);
        m.M = B; m.N = D; m.K = F; m.m_valid = B;
        m.a = {dU, F, B, BcF, false};
        m.b = {w.W1t, F, D, DF, false};
        m.c_gpitch = BcD; m.c0 = t.dS; m.r = t.dZ32; m.inv_scale = inv;
        if ((st = run_train_gemm(c, TE_DRESID, m, nullptr, "dS", s)) != RM_OK) return st;
    }
    {   // dW1 = S^T dU
        ProfScope ps(c, RM_K_BWD_WGRAD, s);
        TrainGemm m = train_gemm_base(c);
        m.M = D; m.N = F; m.K = B; m.m_valid = D;
        m.a = {sl.S, D, B, BcD, true};
        m.b = {dU, F, B, BcF, true};
        m.c_gpitch = DF; m.c0 = gr.dW1; m.inv_scale = inv;
        if ((st = run_train_gemm(c, TE_F32, m, nullptr, "dW1", s)) != RM_OK) return st;
    }
    {
        ProfScope ps(c, RM_K_BWD_ROWS, s);
        const int grid1 = ln1_bwd_grid(B, T, D, c->num_sms);
        float* p_dg1 = t.part1;
        float* p_dbe1 = t.part1 + (size_t)t.grid1 * D;
        RM_CHECK_CUDA(launch_ln1_mix_backward(c->act, sl.Yh, sl.rstd1, t.dS, w.g1, dX, p_dg1, p_dbe1, B, T, D, Bc,
                                              grid1, c->d_err, kWaitTimeoutNs, s),
                      "ln1 + mixing backward");
        if (db1_partials)
            RM_CHECK_CUDA(launch_sum_rows(t.colpart, gr.db1, nullptr, T, colrows, F, s), "db1");
        RM_CHECK_CUDA(launch_sum_rows(p_db2, gr.db2, nullptr, T, nblk, D, s), "db2");
        RM_CHECK_CUDA(launch_sum_rows(p_dg2, t.tmpTD, gr.dln2_gamma, T, nblk, D, s), "dgamma2");
        RM_CHECK_CUDA(launch_sum_rows(p_dbe2, t.tmpTD, gr.dln2_beta, T, nblk, D, s), "dbeta2");
        RM_CHECK_CUDA(launch_sum_rows(p_dg1, gr.dln1_gamma, nullptr, 1, grid1, D, s), "dgamma1");
        RM_CHECK_CUDA(launch_sum_rows(p_dbe1, gr.dln1_beta, nullptr, 1, grid1, D, s), "dbeta1");
    }
    return RM_OK;
}

// The stack's training forward: every layer's activations into its slot; the
// next layer's input X_{n+1} = LN2(Z_n) in float32; pooled from the last Z.
rm_status stack_forward_train_impl(rm_ctx* c, const void* X0, float* pooled, int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    TrainWS& t = c->tw;
    rm_status st;
    t.saved_B = 0;
    for (int n = 0; n < g.L; ++n) {
        if ((st = train_layer_forward(c, n, n, n == 0 ? X0 : t.Xn, n > 0, B, s)) != RM_OK) return st;
        const TrainSlot& sl = t.slots[n];
        {
            ProfScope ps(c, RM_K_ROWSTATS, s);
            RM_CHECK_CUDA(launch_rowstats(c->act, sl.Z, c->rows, B, g.T, g.D, c->Bcap, c->num_sms, s), "row stats");
        }
        if (n + 1 < g.L) {
            ProfScope ps(c, RM_K_LN2_OUT, s);
            RM_CHECK_CUDA(launch_ln2_out(c->act, sl.Z, c->rows, c->layers[n].g2, c->layers[n].be2, t.Xn,
                                         /*out_f32*/ true, B, g.T, g.D, c->Bcap, 1, g.D, g.ln_eps, c->num_sms, s),
                          "ln2 out");
        } else {
            ProfScope ps(c, RM_K_POOL, s);
            RM_CHECK_CUDA(launch_pool(c->act, sl.Z, c->rows, c->layers[n].g2, c->layers[n].be2, pooled, nullptr,
                                      false, B, g.T, g.D, c->Bcap, 1, g.D, g.ln_eps, c->num_sms, c->d_err,
                                      kWaitTimeoutNs, s),
                          "ln2 + pool");
        }
    }
    t.saved_B = B;
    return RM_OK;
}

// The stack's backward from the slots rm_stack_forward_train filled.
rm_status stack_backward_saved_impl(rm_ctx* c, const float* dpooled, float* dX0, const rm_layer_grads* grads, int B,
                                    cudaStream_t s) {
    const rm_config& g = c->cfg;
    TrainWS& t = c->tw;
    rm_status st;
    {
        ProfScope ps(c, RM_K_BWD_ROWS, s);
        RM_CHECK_CUDA(launch_pool_backward(dpooled, t.G0, B, g.T, g.D, s), "pool backward");
    }
    float* gcur = t.G0;
    float* gnext = t.G1;
    t.saved_B = 0;            // the backward consumes Gelu'(U) of every slot
    for (int n = g.L - 1; n >= 0; --n) {
        float* out = n == 0 ? dX0 : gnext;
        if ((st = train_layer_backward(c, n, n, gcur, out, grads[n], B, s)) != RM_OK) return st;
        float* tmp = gcur;
        gcur = gnext;
        gnext = tmp;
    }
    return RM_OK;
}

rm_status check_backward(rm_ctx* c, int B) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (!c->cfg.training) return fail(RM_ERR_UNSUPPORTED, "the context was created without cfg.training");
    for (const auto& l : c->layers)
        if (l.um_bs) return fail(RM_ERR_UNSUPPORTED, "UniMixing layers have no training path");
    return check_batch(c, B);
}

// ---- UniMixing ("UniMixer" section 4.3) ------------------------------------------
long long um_pitch(const rm_ctx* c, int bs) { return ((long long)c->Bcap * bs + 255) / 256 * 256; }

XType caller_xtype(const rm_ctx* c) { return c->act == Act::F32 ? XType::F32 : XType::BF16; }
XType op_xtype(const rm_ctx* c) { return c->act == Act::F32 ? XType::F32 : XType::F16; }

// Local step and global product of layer `layer` for B samples of X (type xt,
// sample-major [B][T][D]) into c->umYt as Y [B][T D] (operand type).
rm_status unimix_global(rm_ctx* c, int layer, const void* X, XType xt, int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    const LayerW& w = c->layers[layer];
    const int bs = w.um_bs;
    const int nb = g.T * g.D / bs;
    const long long Npitch = um_pitch(c, bs);
    const long long Npad = ((long long)B * bs + 255) / 256 * 256;
    RM_CHECK_CUDA(launch_unimix_local(xt, c->act, X, (long long)g.T * g.D, w.umWB, w.umWBt16, c->umH, B, nb, bs,
                                      Npitch, Npad, c->num_sms, c->d_err, kWaitTimeoutNs, s),
                  "unimixing local step");
    TrainGemm m = train_gemm_base(c);
    m.G = 1;
    m.M = nb; m.N = (int)Npad; m.K = nb; m.m_valid = nb;
    m.a = {w.umWGop, nb, nb, 0, false};                    // WG [i][j], K-major
    m.b = {c->umH, (int)Npad, nb, 0, true, Npitch};        // H [j][n], MN-major
    m.c_gpitch = 0; m.c_ld = Npitch;
    m.c0 = c->umYt;
    m.um_bs = bs; m.um_B = B; m.um_L = (long long)g.T * g.D;
    return run_train_gemm(c, TE_F16T, m, nullptr, "unimixing global product", s);
}

// S = LN1(X + UniMixing(X)) for layer `layer` (its mixing step, in place of
// mix + LN1).  X: the layer input in type xt, sample-major.
rm_status unimix_mix_ln1(rm_ctx* c, int layer, const void* X, XType xt, int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    const LayerW& w = c->layers[layer];
    ProfScope ps(c, RM_K_UNIMIX, s);
    rm_status st = unimix_global(c, layer, X, xt, B, s);
    if (st != RM_OK) return st;
    RM_CHECK_CUDA(launch_unimix_ln1(xt, c->act, X, c->umYt, c->S, w.g1, w.be1, B, g.T, g.D, c->Bcap, g.ln_eps,
                                    c->num_sms, s),
                  "unimixing residual + ln1");
    return RM_OK;
}

}  // namespace

cudaError_t rm::device_alloc(void** p, size_t bytes) {
    *p = nullptr;
    AllocBook& b = book();
    {
        std::lock_guard<std::mutex> lk(b.mu);
        read_fault_env(b);
        b.last_injected = false;
        if (b.fail_after == 0) {
            b.fail_after = -1;          // one failure per arming
            b.last_injected = true;
            return cudaErrorMemoryAllocation;
        }
        if (b.fail_after > 0) --b.fail_after;
    }
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        *p = nullptr;
        return e;
    }
    std::lock_guard<std::mutex> lk(b.mu);
    b.live[*p] = bytes;
    b.made += 1;
    b.live_bytes += (long long)bytes;
    return cudaSuccess;
}

void rm::device_free(void* p) {
    if (!p) return;
    cudaFree(p);
    AllocBook& b = book();
    std::lock_guard<std::mutex> lk(b.mu);
    auto it = b.live.find(p);
    if (it != b.live.end()) {
        b.live_bytes -= (long long)it->second;
        b.live.erase(it);
    }
}

// =============================================================================
// Public entry points
// =============================================================================
extern "C" {

int rm_abi_version(void) { return RM_ABI_VERSION; }

const char* rm_last_error(void) { return g_last_error.c_str(); }

rm_status rm_create(const rm_config* cfg, const rm_layer_params* layers, int device, rm_ctx** out) {
    g_last_error.clear();
    if (!out) return fail(RM_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    rm_status st = validate_cfg(cfg);
    if (st != RM_OK) return st;
    if (!layers) return fail(RM_ERR_INVALID_ARG, "layers is NULL");
    int ndev = 0;
    RM_CHECK_CUDA(cudaGetDeviceCount(&ndev), "cudaGetDeviceCount");
    if (device < 0 || device >= ndev) return fail(RM_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, ndev);
    RM_CHECK_CUDA(cudaSetDevice(device), "cudaSetDevice");
    cudaDeviceProp prop;
    RM_CHECK_CUDA(cudaGetDeviceProperties(&prop, device), "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(RM_ERR_UNSUPPORTED, "this library is built for sm_103a only (device is sm_%d%d)", prop.major,
                    prop.minor);

    rm_ctx* c = new rm_ctx();
    c->cfg = *cfg;
    c->device = device;
    c->num_sms = prop.multiProcessorCount;
    c->act = cfg->dtype == RM_F32 ? Act::F32 : Act::BF16;
    c->esz = act_size(c->act);
    c->F = cfg->k * cfg->D;
    const bool tc_ok = c->act == Act::BF16 && tc_supported(cfg->D, c->F);
    if (cfg->gemm_path == RM_PATH_TCGEN05 && !tc_ok) {
        delete c;
        return fail(RM_ERR_UNSUPPORTED, "tcgen05 path needs bf16 and D, kD multiples of 64");
    }
    c->use_tc = tc_ok && cfg->gemm_path != RM_PATH_SIMT;
    c->cw = c->use_tc ? tc_stats_chunk_width(cfg->D) : cfg->D;
    c->nchunk = cfg->D / c->cw;
    c->Bcap = cfg->max_batch;

    const size_t T = cfg->T, D = cfg->D, F = c->F, Bc = c->Bcap;
    if ((st = dmalloc(c, &c->S, T * Bc * D * c->esz, &c->ws_bytes)) != RM_OK ||
        (st = dmalloc(c, &c->Hid, T * Bc * F * c->esz, &c->ws_bytes)) != RM_OK ||
        (st = dmalloc(c, &c->Z, T * Bc * D * op_size(c->act), &c->ws_bytes)) != RM_OK ||
        (st = dmalloc(c, (void**)&c->stats, T * Bc * (size_t)c->nchunk * sizeof(float2), &c->ws_bytes)) != RM_OK ||
        (st = dmalloc(c, (void**)&c->rows, T * Bc * sizeof(float2), &c->ws_bytes)) != RM_OK ||
        (st = dmalloc(c, (void**)&c->d_err, sizeof(int), nullptr)) != RM_OK ||
        (st = dmalloc(c, (void**)&c->d_flag, sizeof(int), nullptr)) != RM_OK) {
        free_ctx(c);
        return st;
    }
    if (c->use_tc) {
        const size_t ndep = T * (size_t)((Bc + 255) / 256);
        if ((st = dmalloc(c, (void**)&c->dep_cnt, ndep * sizeof(unsigned), nullptr)) != RM_OK) {
            free_ctx(c);
            return st;
        }
        cudaError_t e = cudaMemset(c->dep_cnt, 0, ndep * sizeof(unsigned));
        if (e != cudaSuccess) {
            free_ctx(c);
            return cuda_fail(e, "clear layer counters");
        }
    }
    if (cfg->moe_layer_mask != 0 &&
        (st = dmalloc(c, (void**)&c->V, T * Bc * D * 4, &c->ws_bytes)) != RM_OK) {
        free_ctx(c);
        return st;
    }
    if (cfg->n_experts > 0) {
        MoeShape ms{c->act, cfg->T, cfg->D, cfg->n_experts, cfg->expert_hidden};
        cudaError_t e = moe_alloc_workspace(ms, c->Bcap, c->moe_ws, &c->ws_bytes);
        if (e != cudaSuccess) {
            free_ctx(c);
            return cuda_fail(e, "MoE workspace");
        }
    }
    cudaMemset(c->d_err, 0, sizeof(int));
    cudaMemset(c->d_flag, 0, sizeof(int));
    c->layers.resize(cfg->L);
    for (int n = 0; n < cfg->L; ++n) {
        st = pack_layer(c, layers[n], c->layers[n], 0);
        if (st != RM_OK) {
            free_ctx(c);
            return st;
        }
    }
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_ctx(c);
        return cuda_fail(e, "rm_create");
    }
    *out = c;
    return RM_OK;
}

rm_status rm_destroy(rm_ctx* ctx) {
    if (!ctx) return RM_OK;
    free_ctx(ctx);
    return RM_OK;
}

rm_status rm_block_forward(rm_ctx* c, int layer, const void* X_in, void* X_out, void* S_out, rm_dtype out_dtype, int B,
                           void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (layer < 0 || layer >= c->cfg.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    if ((st = check_batch(c, B)) != RM_OK) return st;
    bool out_f32 = false;
    if ((st = check_out_dtype(c, out_dtype, &out_f32)) != RM_OK) return st;
    if (!X_in || !X_out) return fail(RM_ERR_INVALID_ARG, "X_in / X_out is NULL");
    if (!aligned16(X_in) || !aligned16(X_out) || (S_out && !aligned16(S_out)))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    const size_t in_bytes = (size_t)B * c->cfg.T * c->cfg.D * c->esz;
    const size_t out_bytes = (size_t)B * c->cfg.T * c->cfg.D * (out_f32 ? 4 : c->esz);
    const char* xi = (const char*)X_in;
    const char* xo = (const char*)X_out;
    if (xi < xo + out_bytes && xo < xi + in_bytes) return fail(RM_ERR_INVALID_ARG, "X_in and X_out overlap");
    cudaSetDevice(c->device);
    cudaStream_t s = as_stream(stream);
    const rm_config& g = c->cfg;
    if (c->layers[layer].um_bs) {
        if ((st = unimix_mix_ln1(c, layer, X_in, caller_xtype(c), B, s)) != RM_OK) return st;
    } else {
        MixLnArgs a = mix_args(c, layer, B);
        a.X = X_in;
        ProfScope ps(c, RM_K_MIX_LN1, s);
        RM_CHECK_CUDA(launch_mix_ln1(c->act, false, a, c->num_sms, s), "mix+ln1");
    }
    if (S_out) {
        ProfScope ps(c, RM_K_MISC, s);
        RM_CHECK_CUDA(launch_token_to_sample(c->act, c->S, S_out, out_f32, B, g.T, g.D, c->Bcap, s), "copy S");
    }
    if ((st = run_pffn(c, layer, B, s)) != RM_OK) return st;
    ProfScope ps(c, RM_K_LN2_OUT, s);
    RM_CHECK_CUDA(launch_ln2_out(c->act, c->Z, c->ln2_st, c->layers[layer].g2, c->layers[layer].be2, X_out, out_f32,
                                 B, g.T, g.D, c->Bcap, c->ln2_nchunk, c->ln2_cw, g.ln_eps, c->num_sms,
                                 s),
                  "ln2 out");
    return RM_OK;
}

rm_status rm_stack_forward(rm_ctx* c, const void* X0, float* pooled, void* XL, rm_dtype xl_dtype, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if ((st = check_batch(c, B)) != RM_OK) return st;
    bool xl_f32 = false;
    if ((st = check_out_dtype(c, xl_dtype, &xl_f32)) != RM_OK) return st;
    if (!X0 || !pooled) return fail(RM_ERR_INVALID_ARG, "X0 / pooled is NULL");
    if (!aligned16(X0) || !aligned16(pooled) || (XL && !aligned16(XL)))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    return stack_device(c, X0, pooled, XL, xl_f32, B, as_stream(stream));
}

rm_status rm_stack_forward_host_async(rm_ctx* c, const void* X0_host, float* pooled_host, int B, void* stream,
                                      long long* ticket) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!X0_host || !pooled_host || !ticket) return fail(RM_ERR_INVALID_ARG, "X0_host / pooled_host / ticket is NULL");
    cudaSetDevice(c->device);
    const rm_config& g = c->cfg;
    const size_t row_in = (size_t)g.T * g.D * c->esz, row_out = (size_t)g.D * 4;
    if ((st = copy_streams(c)) != RM_OK) return st;
    const int k = (int)(c->h_next & 1);
    if ((st = ensure(c, &c->hx_dev[k], (size_t)c->Bcap * row_in, &c->ws_bytes)) != RM_OK) return st;
    if ((st = ensure(c, (void**)&c->hp_dev[k], (size_t)c->Bcap * row_out, &c->ws_bytes)) != RM_OK) return st;
    if (!c->hx_in[k]) {
        RM_CHECK_CUDA(cudaEventCreateWithFlags(&c->hx_in[k], cudaEventDisableTiming), "event");
        RM_CHECK_CUDA(cudaEventCreateWithFlags(&c->hx_done[k], cudaEventDisableTiming), "event");
        RM_CHECK_CUDA(cudaEventCreateWithFlags(&c->hx_out[k], cudaEventDisableTiming), "event");
    }
    if (c->h_slot[k] >= 0) {            // the batch two calls back still holds this slot
        RM_CHECK_CUDA(cudaEventSynchronize(c->hx_out[k]), "wait for the slot's previous batch");
        c->h_slot[k] = -1;
    }
    cudaStream_t s = as_stream(stream);
    // the copy runs on its own stream while the previous batch computes on `stream`
    RM_CHECK_CUDA(cudaMemcpyAsync(c->hx_dev[k], X0_host, (size_t)B * row_in, cudaMemcpyHostToDevice, c->s_in),
                  "H2D X0");
    RM_CHECK_CUDA(cudaEventRecord(c->hx_in[k], c->s_in), "event");
    RM_CHECK_CUDA(cudaStreamWaitEvent(s, c->hx_in[k], 0), "wait");
    if ((st = stack_device(c, c->hx_dev[k], c->hp_dev[k], nullptr, false, B, s)) != RM_OK) return st;
    RM_CHECK_CUDA(cudaEventRecord(c->hx_done[k], s), "event");
    RM_CHECK_CUDA(cudaStreamWaitEvent(c->s_out, c->hx_done[k], 0), "wait");
    RM_CHECK_CUDA(cudaMemcpyAsync(pooled_host, c->hp_dev[k], (size_t)B * row_out, cudaMemcpyDeviceToHost, c->s_out),
                  "D2H pooled");
    RM_CHECK_CUDA(cudaEventRecord(c->hx_out[k], c->s_out), "event");
    c->h_slot[k] = c->h_next;
    *ticket = c->h_next++;
    return RM_OK;
}

rm_status rm_host_wait(rm_ctx* c, long long ticket) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (ticket < 0 || ticket >= c->h_next)
        return fail(RM_ERR_INVALID_ARG, "ticket %lld was not issued by this context", ticket);
    const int k = (int)(ticket & 1);
    if (c->h_slot[k] != ticket) return RM_OK;      // already waited for, or its slot has been reused since
    cudaSetDevice(c->device);
    RM_CHECK_CUDA(cudaEventSynchronize(c->hx_out[k]), "wait for the batch");
    c->h_slot[k] = -1;
    return RM_OK;
}

rm_status rm_stack_forward_host(rm_ctx* c, const void* X0_host, float* pooled_host, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!X0_host || !pooled_host) return fail(RM_ERR_INVALID_ARG, "X0_host / pooled_host is NULL");
    cudaSetDevice(c->device);
    const rm_config& g = c->cfg;
    if ((st = ensure(c, &c->X0_dev, (size_t)c->Bcap * g.T * g.D * c->esz, &c->ws_bytes)) != RM_OK) return st;
    if ((st = ensure(c, (void**)&c->pooled_dev, (size_t)c->Bcap * g.D * 4, &c->ws_bytes)) != RM_OK) return st;
    cudaStream_t s = as_stream(stream);
    const size_t row_in = (size_t)g.T * g.D * c->esz, row_out = (size_t)g.D * 4;
    char* x_dev = static_cast<char*>(c->X0_dev);
    const char* x_host = static_cast<const char*>(X0_host);
    // Large batches run as three growing chunks, B/8, 3B/8 and the rest (whole
    // multiples of 256 samples, the CTA-pair tile height): chunk i + 1 is copied
    // in on one stream while chunk i computes on `stream`, and each chunk's
    // pooled rows go back on a third; the workspace is reused chunk after chunk
    // (the compute is serial).  Only the first, small chunk's copy is exposed,
    // and the two large chunks run near the full batch's GEMM efficiency.  (Four
    // equal chunks measured 7.5% slower compute at the 1B shape and exposed a
    // copy twice as long.)
    int bounds[kHostChunksMax + 1] = {0};
    int nchunks = 1;
    bounds[1] = B;
    if (B >= 2 * kHostChunkMin) {
        const int c0 = (B / 8 + 255) / 256 * 256;
        const int c1 = (3 * B / 8 + 255) / 256 * 256;
        if (c0 + c1 < B) {
            bounds[1] = c0;
            bounds[2] = c0 + c1;
            bounds[3] = B;
            nchunks = 3;
        }
    }
    if (nchunks == 1) {
        {
            ProfScope ps(c, RM_K_MISC, s);
            RM_CHECK_CUDA(cudaMemcpyAsync(c->X0_dev, X0_host, (size_t)B * row_in, cudaMemcpyHostToDevice, s), "H2D X0");
        }
        if ((st = stack_device(c, c->X0_dev, c->pooled_dev, nullptr, false, B, s)) != RM_OK) return st;
        {
            ProfScope ps(c, RM_K_MISC, s);
            RM_CHECK_CUDA(cudaMemcpyAsync(pooled_host, c->pooled_dev, (size_t)B * row_out, cudaMemcpyDeviceToHost, s),
                          "D2H pooled");
        }
        RM_CHECK_CUDA(cudaStreamSynchronize(s), "stream sync");
        return RM_OK;
    }
    if ((st = copy_streams(c)) != RM_OK) return st;
    // the staging buffers may still be read by an earlier call's work on `stream`
    RM_CHECK_CUDA(cudaEventRecord(c->ev_done[0], s), "event");
    RM_CHECK_CUDA(cudaStreamWaitEvent(c->s_in, c->ev_done[0], 0), "wait");
    for (int i = 0; i < nchunks; ++i) {
        const int b0 = bounds[i], bn = bounds[i + 1] - bounds[i];
        RM_CHECK_CUDA(cudaMemcpyAsync(x_dev + (size_t)b0 * row_in, x_host + (size_t)b0 * row_in, (size_t)bn * row_in,
                                      cudaMemcpyHostToDevice, c->s_in),
                      "H2D X0 chunk");
        RM_CHECK_CUDA(cudaEventRecord(c->ev_in[i], c->s_in), "event");
    }
    for (int i = 0; i < nchunks; ++i) {
        const int b0 = bounds[i], bn = bounds[i + 1] - bounds[i];
        RM_CHECK_CUDA(cudaStreamWaitEvent(s, c->ev_in[i], 0), "wait");
        if ((st = stack_device(c, x_dev + (size_t)b0 * row_in, c->pooled_dev + (size_t)b0 * g.D, nullptr, false, bn, s)) !=
            RM_OK)
            return st;
        RM_CHECK_CUDA(cudaEventRecord(c->ev_done[i], s), "event");
        RM_CHECK_CUDA(cudaStreamWaitEvent(c->s_out, c->ev_done[i], 0), "wait");
        RM_CHECK_CUDA(cudaMemcpyAsync(pooled_host + (size_t)b0 * g.D, c->pooled_dev + (size_t)b0 * g.D,
                                      (size_t)bn * row_out, cudaMemcpyDeviceToHost, c->s_out),
                      "D2H pooled chunk");
    }
    RM_CHECK_CUDA(cudaStreamSynchronize(c->s_out), "stream sync");
    RM_CHECK_CUDA(cudaStreamSynchronize(s), "stream sync");
    return RM_OK;
}

rm_status rm_moe_pffn_forward(rm_ctx* c, int layer, const void* S, float* V_out, float* gates, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (c->cfg.n_experts <= 0) return fail(RM_ERR_UNSUPPORTED, "context was created without experts");
    if (layer < 0 || layer >= c->cfg.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!S || !V_out) return fail(RM_ERR_INVALID_ARG, "S / V_out is NULL");
    if (!aligned16(S) || !aligned16(V_out) || (gates && !aligned16(gates)))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    cudaStream_t s = as_stream(stream);
    const rm_config& g = c->cfg;
    MoeLaunch ml{c->act, S, /*S sample-major*/ true, g.T, g.D, g.n_experts, g.expert_hidden, B, c->Bcap, c->num_sms, c->d_err};
    cudaError_t e = moe_forward(ml, c->layers[layer].moe, c->moe_ws, V_out, /*V token-major*/ false, gates, s,
                                [&](int kind) { return (void*)new ProfScope(c, kind, s); },
                                [](void* p) { delete (ProfScope*)p; });
    if (e != cudaSuccess) return cuda_fail(e, "moe pffn");
    return RM_OK;
}

rm_status rm_block_backward(rm_ctx* c, int layer, const void* X_in, const float* dX_out, float* dX_in,
                            const rm_layer_grads* grads, int B, void* stream) {
    rm_status st;
    if ((st = check_backward(c, B)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (layer < 0 || layer >= g.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (g.moe_layer_mask & (1u << layer)) return fail(RM_ERR_UNSUPPORTED, "the backward pass covers dense layers");
    if (!X_in || !dX_out || !dX_in) return fail(RM_ERR_INVALID_ARG, "X_in / dX_out / dX_in is NULL");
    if (!aligned16(X_in) || !aligned16(dX_out) || !aligned16(dX_in))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    if ((st = check_grads(grads)) != RM_OK) return st;
    const size_t gb = (size_t)B * g.T * g.D * 4;
    const char* gi = (const char*)dX_out;
    const char* go = (const char*)dX_in;
    if (gi < go + gb && go < gi + gb) return fail(RM_ERR_INVALID_ARG, "dX_out and dX_in overlap");
    cudaSetDevice(c->device);
    if ((st = train_ws_ready(c, 1, false)) != RM_OK) return st;
    cudaStream_t s = as_stream(stream);
    c->tw.saved_B = 0;        // slot 0 is reused
    if ((st = train_layer_forward(c, layer, 0, X_in, false, B, s)) != RM_OK) return st;
    return train_layer_backward(c, layer, 0, dX_out, dX_in, *grads, B, s);
}

rm_status rm_stack_forward_train(rm_ctx* c, const void* X0, float* pooled, int B, void* stream) {
    rm_status st;
    if ((st = check_backward(c, B)) != RM_OK) return st;
    if (c->cfg.moe_layer_mask != 0) return fail(RM_ERR_UNSUPPORTED, "the training path covers dense layers");
    if (!X0 || !pooled) return fail(RM_ERR_INVALID_ARG, "X0 / pooled is NULL");
    if (!aligned16(X0) || !aligned16(pooled)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    if ((st = train_ws_ready(c, c->cfg.L, true)) != RM_OK) return st;
    return stack_forward_train_impl(c, X0, pooled, B, as_stream(stream));
}

rm_status rm_stack_backward_saved(rm_ctx* c, const float* dpooled, float* dX0, const rm_layer_grads* grads, int B,
                                  void* stream) {
    rm_status st;
    if ((st = check_backward(c, B)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (!dpooled || !dX0) return fail(RM_ERR_INVALID_ARG, "dpooled / dX0 is NULL");
    if (!aligned16(dpooled) || !aligned16(dX0)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    if (!grads) return fail(RM_ERR_INVALID_ARG, "grads is NULL");
    for (int n = 0; n < g.L; ++n)
        if ((st = check_grads(grads + n)) != RM_OK) return st;
    if (c->tw.saved_B == 0)
        return fail(RM_ERR_INVALID_ARG, "no saved activations: call rm_stack_forward_train first (once per backward)");
    if (c->tw.saved_B != B)
        return fail(RM_ERR_INVALID_ARG, "B (%d) differs from the training forward's batch (%d)", B, c->tw.saved_B);
    cudaSetDevice(c->device);
    return stack_backward_saved_impl(c, dpooled, dX0, grads, B, as_stream(stream));
}

rm_status rm_stack_backward(rm_ctx* c, const void* X0, const float* dpooled, float* dX0, const rm_layer_grads* grads,
                            int B, void* stream) {
    rm_status st;
    if ((st = check_backward(c, B)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (g.moe_layer_mask != 0) return fail(RM_ERR_UNSUPPORTED, "the backward pass covers dense layers");
    if (!X0 || !dpooled || !dX0) return fail(RM_ERR_INVALID_ARG, "X0 / dpooled / dX0 is NULL");
    if (!aligned16(X0) || !aligned16(dpooled) || !aligned16(dX0))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    if (!grads) return fail(RM_ERR_INVALID_ARG, "grads is NULL");
    for (int n = 0; n < g.L; ++n)
        if ((st = check_grads(grads + n)) != RM_OK) return st;
    cudaSetDevice(c->device);
    if ((st = train_ws_ready(c, g.L, true)) != RM_OK) return st;
    cudaStream_t s = as_stream(stream);
    if ((st = stack_forward_train_impl(c, X0, c->tw.pooled, B, s)) != RM_OK) return st;
    return stack_backward_saved_impl(c, dpooled, dX0, grads, B, s);
}

rm_status rm_head_forward(const float* pooled, const float* w, float b, const float* y, float* p, float* loss,
                          float* dpooled, int B, int D, int mean_loss, void* stream) {
    if (B < 1 || D < 1) return fail(RM_ERR_INVALID_ARG, "B and D must be positive");
    if (!pooled || !w) return fail(RM_ERR_INVALID_ARG, "pooled / w is NULL");
    if (!y && (loss || dpooled)) return fail(RM_ERR_INVALID_ARG, "loss and dpooled need the labels y");
    if (!p && !loss && !dpooled) return fail(RM_ERR_INVALID_ARG, "no output requested");
    if (!aligned16(pooled) || !aligned16(w) || (dpooled && !aligned16(dpooled)))
        return fail(RM_ERR_INVALID_ARG, "pooled, w and dpooled must be 16-byte aligned");
    if (!std::isfinite(b)) return fail(RM_ERR_INVALID_ARG, "b must be finite");
    const float gscale = mean_loss ? 1.0f / (float)B : 1.0f;
    RM_CHECK_CUDA(launch_head(pooled, w, b, y, p, loss, dpooled, gscale, B, D, as_stream(stream)), "head");
    return RM_OK;
}

rm_status rm_set_tokenizer(rm_ctx* c, const void* W, const void* bias, int d) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (!W || !bias) return fail(RM_ERR_INVALID_ARG, "W / bias is NULL");
    if (d < 1) return fail(RM_ERR_INVALID_ARG, "d must be positive");
    const rm_config& g = c->cfg;
    cudaSetDevice(c->device);
    device_free(c->Wtok); device_free(c->btok); device_free(c->Etok);
    c->Wtok = nullptr; c->btok = nullptr; c->Etok = nullptr; c->tok_d = 0;
    const long long n = (long long)g.T * d * g.D;
    if ((st = dmalloc(c, &c->Wtok, (size_t)n * c->esz, &c->weight_bytes)) != RM_OK) return st;
    if ((st = dmalloc(c, (void**)&c->btok, (size_t)g.T * g.D * 4, &c->weight_bytes)) != RM_OK) return st;
    if (c->act == Act::F32)
        RM_CHECK_CUDA(cudaMemcpy(c->Wtok, W, (size_t)n * 4, cudaMemcpyDeviceToDevice), "copy tokenizer W");
    else {
        RM_CHECK_CUDA(launch_bf16_to_f16(W, c->Wtok, n, 0), "copy tokenizer W");
        if ((st = dmalloc(c, &c->Etok, (size_t)c->Bcap * g.T * d * 2, &c->ws_bytes)) != RM_OK) return st;
    }
    RM_CHECK_CUDA(launch_to_f32(c->act, bias, c->btok, (size_t)g.T * g.D, 0), "copy tokenizer bias");
    RM_CHECK_CUDA(cudaDeviceSynchronize(), "rm_set_tokenizer");
    c->tok_d = d;
    return RM_OK;
}

rm_status rm_set_unimixing(rm_ctx* c, int layer, const float* WG, const float* WB, int bs, float tau, int iters,
                           void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (layer < 0 || layer >= g.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!WG || !WB) return fail(RM_ERR_INVALID_ARG, "WG / WB is NULL");
    const long long L = (long long)g.T * g.D;
    if (bs < 1 || L % bs != 0) return fail(RM_ERR_INVALID_ARG, "bs (%d) must divide T * D (%lld)", bs, L);
    if (!(tau > 0.f) || !std::isfinite(tau)) return fail(RM_ERR_INVALID_ARG, "tau must be positive and finite");
    if (iters < 0) return fail(RM_ERR_INVALID_ARG, "iters must be >= 0");
    if (g.D > 48 * 32) return fail(RM_ERR_UNSUPPORTED, "UniMixing rows support D <= 1536");
    const int nb = (int)(L / bs);
    cudaSetDevice(c->device);
    cudaStream_t s = as_stream(stream);
    RM_CHECK_CUDA(cudaStreamSynchronize(s), "rm_set_unimixing (drain the stream)");
    LayerW& w = c->layers[layer];
    if (w.umWGop != w.umWG32) device_free(w.umWGop);
    device_free(w.umWG32); device_free(w.umWB); device_free(w.umWBt16);
    w.umWG32 = nullptr; w.umWGop = nullptr; w.umWB = nullptr; w.umWBt16 = nullptr; w.um_bs = 0;
    const size_t nG = (size_t)nb * nb, nB = (size_t)nb * bs * bs;
    if ((st = dmalloc(c, (void**)&w.umWG32, nG * 4, &c->weight_bytes)) != RM_OK) return st;
    if ((st = dmalloc(c, (void**)&w.umWB, nB * 4, &c->weight_bytes)) != RM_OK) return st;
    if (c->act == Act::F32)
        w.umWGop = w.umWG32;
    else if ((st = dmalloc(c, &w.umWGop, nG * 2, &c->weight_bytes)) != RM_OK)
        return st;
    if (c->act != Act::F32 && unimix_local_mma_ok(bs) &&
        (st = dmalloc(c, &w.umWBt16, nB * 2, &c->weight_bytes)) != RM_OK)
        return st;
    // workspace for the largest pitch so far
    const size_t hy = (size_t)nb * (size_t)um_pitch(c, bs) * op_size(c->act);
    if (hy > c->um_bytes) {
        device_free(c->umH); device_free(c->umYt);
        c->umH = nullptr; c->umYt = nullptr; c->um_bytes = 0;
        if ((st = dmalloc(c, &c->umH, hy, &c->ws_bytes)) != RM_OK) return st;
        if ((st = dmalloc(c, &c->umYt, hy, &c->ws_bytes)) != RM_OK) return st;
        c->um_bytes = hy;
    }
    if (!c->umX && (st = dmalloc(c, &c->umX, (size_t)c->Bcap * L * op_size(c->act), &c->ws_bytes)) != RM_OK)
        return st;
    // Sinkhorn-Knopp scratch, freed again below
    float *C = nullptr, *f = nullptr, *gv = nullptr;
    const size_t nmax = nG > nB ? nG : nB;
    const size_t vmax = (size_t)nb * (size_t)(bs > 1 ? bs : 1) > (size_t)nb ? (size_t)nb * bs : (size_t)nb;
    if ((st = dmalloc(c, (void**)&C, nmax * 4, nullptr)) != RM_OK) return st;
    if ((st = dmalloc(c, (void**)&f, vmax * 4, nullptr)) != RM_OK || (st = dmalloc(c, (void**)&gv, vmax * 4, nullptr)) != RM_OK) {
        device_free(C); device_free(f);
        return st;
    }
    cudaError_t e = launch_sinkhorn(WG, 1, nb, tau, iters, C, f, gv, w.umWG32, c->act == Act::F32 ? nullptr : w.umWGop, s);
    if (e == cudaSuccess) e = launch_sinkhorn(WB, nb, bs, tau, iters, C, f, gv, w.umWB, nullptr, s);
    if (e == cudaSuccess && w.umWBt16) e = launch_unimix_pack_wb(w.umWB, w.umWBt16, nb, bs, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    device_free(C); device_free(f); device_free(gv);
    if (e != cudaSuccess) return cuda_fail(e, "rm_set_unimixing (Sinkhorn-Knopp)");
    w.um_bs = bs;
    return RM_OK;
}

rm_status rm_unimixing_weights(rm_ctx* c, int layer, float* WG_out, float* WB_out, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (layer < 0 || layer >= g.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    const LayerW& w = c->layers[layer];
    if (!w.um_bs) return fail(RM_ERR_INVALID_ARG, "layer %d uses TokenMixing (no rm_set_unimixing)", layer);
    if (!WG_out && !WB_out) return fail(RM_ERR_INVALID_ARG, "WG_out and WB_out are NULL");
    const size_t nb = (size_t)g.T * g.D / w.um_bs;
    cudaSetDevice(c->device);
    cudaStream_t s = as_stream(stream);
    if (WG_out) RM_CHECK_CUDA(cudaMemcpyAsync(WG_out, w.umWG32, nb * nb * 4, cudaMemcpyDeviceToDevice, s), "copy WG");
    if (WB_out)
        RM_CHECK_CUDA(cudaMemcpyAsync(WB_out, w.umWB, nb * w.um_bs * w.um_bs * 4, cudaMemcpyDeviceToDevice, s),
                      "copy WB");
    return RM_OK;
}

rm_status rm_unimixing(rm_ctx* c, int layer, const void* X, void* Y, rm_dtype out_dtype, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    bool out_f32 = false;
    if ((st = check_out_dtype(c, out_dtype, &out_f32)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (layer < 0 || layer >= g.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!c->layers[layer].um_bs) return fail(RM_ERR_INVALID_ARG, "layer %d uses TokenMixing (no rm_set_unimixing)", layer);
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!X || !Y) return fail(RM_ERR_INVALID_ARG, "X / Y is NULL");
    if (!aligned16(X) || !aligned16(Y)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    cudaStream_t s = as_stream(stream);
    ProfScope ps(c, RM_K_UNIMIX, s);
    if ((st = unimix_global(c, layer, X, caller_xtype(c), B, s)) != RM_OK) return st;
    RM_CHECK_CUDA(launch_unimix_out(c->act, c->umYt, Y, out_f32, (long long)B * g.T * g.D, s), "unimixing output");
    return RM_OK;
}

namespace {
rm_status tokenize_impl(rm_ctx* c, const void* E, void* X0, int B, cudaStream_t s) {
    const rm_config& g = c->cfg;
    const int T = g.T, D = g.D, d = c->tok_d;
    ProfScope ps(c, RM_K_TOKENIZE, s);
    const void* Eop = E;
    if (c->act != Act::F32) {
        RM_CHECK_CUDA(launch_bf16_to_f16(E, c->Etok, (long long)B * T * d, s), "embeddings to fp16");
        Eop = c->Etok;
    }
    TrainGemm m = train_gemm_base(c);
    m.M = B; m.N = D; m.K = d; m.m_valid = B;
    m.a = {Eop, d, B, d, false, (long long)T * d};        // slice t of row b: E[b][t d .. t d + d)
    m.b = {c->Wtok, D, d, (long long)d * D, true};        // W_t [d][D]
    m.c_gpitch = D; m.c_ld = (long long)T * D;            // X0[b][t][:]
    m.c0 = X0; m.bias = c->btok;
    return run_train_gemm(c, TE_BIAS_IO, m, nullptr, "tokenize", s);
}
}  // namespace

rm_status rm_tokenize(rm_ctx* c, const void* E, void* X0, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (c->tok_d == 0) return fail(RM_ERR_INVALID_ARG, "no tokenizer: call rm_set_tokenizer first");
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!E || !X0) return fail(RM_ERR_INVALID_ARG, "E / X0 is NULL");
    if (!aligned16(E) || !aligned16(X0)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    return tokenize_impl(c, E, X0, B, as_stream(stream));
}

rm_status rm_tokenize_backward(rm_ctx* c, const void* E, const float* dX0, float* dE, float* dW, float* db, int B,
                               void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (c->tok_d == 0) return fail(RM_ERR_INVALID_ARG, "no tokenizer: call rm_set_tokenizer first");
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!E || !dX0 || !dW || !db) return fail(RM_ERR_INVALID_ARG, "E / dX0 / dW / db is NULL");
    if (!aligned16(E) || !aligned16(dX0) || !aligned16(dW) || !aligned16(db) || (dE && !aligned16(dE)))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    const rm_config& g = c->cfg;
    const int T = g.T, D = g.D, d = c->tok_d;
    constexpr int kTokParts = 16;
    cudaStream_t s = as_stream(stream);
    ProfScope ps(c, RM_K_TOKENIZE, s);
    const void* Eop = E;
    const void* Gop = dX0;
    const float* inv = nullptr;
    if (c->act != Act::F32) {
        if ((st = ensure(c, &c->dX0h, (size_t)c->Bcap * T * D * 2, &c->ws_bytes)) != RM_OK) return st;
        if ((st = ensure(c, (void**)&c->tok_part, (size_t)T * kTokParts * 4, &c->ws_bytes)) != RM_OK) return st;
        if ((st = ensure(c, (void**)&c->tok_inv, (size_t)T * 4, &c->ws_bytes)) != RM_OK) return st;
        RM_CHECK_CUDA(launch_bf16_to_f16(E, c->Etok, (long long)B * T * d, s), "embeddings to fp16");
        RM_CHECK_CUDA(launch_token_grad_scale(dX0, c->tok_part, kTokParts, c->tok_inv, c->dX0h, B, T, D, s),
                      "token gradient scale");
        Eop = c->Etok;
        Gop = c->dX0h;
        inv = c->tok_inv;
    }
    // dW_t = E_t^T dX0_t: both operands MN-major, K = the batch
    TrainGemm m = train_gemm_base(c);
    m.M = d; m.N = D; m.K = B; m.m_valid = d;
    m.a = {Eop, d, B, d, true, (long long)T * d};
    m.b = {Gop, D, B, D, true, (long long)T * D};
    m.c_gpitch = (long long)d * D; m.c0 = dW; m.inv_scale = inv;
    if ((st = run_train_gemm(c, TE_F32, m, nullptr, "tokenizer dW", s)) != RM_OK) return st;
    if (dE) {   // dE slice t = dX0_t W_t^T
        m = train_gemm_base(c);
        m.M = B; m.N = d; m.K = D; m.m_valid = B;
        m.a = {Gop, D, B, D, false, (long long)T * D};
        m.b = {c->Wtok, D, d, (long long)d * D, false};
        m.c_gpitch = d; m.c_ld = (long long)T * d; m.c0 = dE; m.inv_scale = inv;
        if ((st = run_train_gemm(c, TE_F32, m, nullptr, "tokenizer dE", s)) != RM_OK) return st;
    }
    RM_CHECK_CUDA(launch_token_colsum(dX0, db, B, T, D, s), "tokenizer db");
    return RM_OK;
}

rm_status rm_score(rm_ctx* c, const void* E, const float* head_w, float head_b, float* p, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (c->tok_d == 0) return fail(RM_ERR_INVALID_ARG, "no tokenizer: call rm_set_tokenizer first");
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!E || !head_w || !p) return fail(RM_ERR_INVALID_ARG, "E / head_w / p is NULL");
    if (!aligned16(E) || !aligned16(head_w)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    if (c->cfg.moe_layer_mask != 0) return fail(RM_ERR_UNSUPPORTED, "rm_score runs dense stacks");
    cudaSetDevice(c->device);
    const rm_config& g = c->cfg;
    if ((st = ensure(c, &c->X0ws, (size_t)c->Bcap * g.T * g.D * c->esz, &c->ws_bytes)) != RM_OK) return st;
    if ((st = ensure(c, (void**)&c->pooled_ws, (size_t)c->Bcap * g.D * 4, &c->ws_bytes)) != RM_OK) return st;
    cudaStream_t s = as_stream(stream);
    if ((st = tokenize_impl(c, E, c->X0ws, B, s)) != RM_OK) return st;
    if ((st = stack_device(c, c->X0ws, c->pooled_ws, nullptr, false, B, s)) != RM_OK) return st;
    ProfScope ps(c, RM_K_HEAD, s);
    RM_CHECK_CUDA(launch_head(c->pooled_ws, head_w, head_b, nullptr, p, nullptr, nullptr, 1.0f, B, g.D, s), "head");
    return RM_OK;
}

rm_status rm_debug_gelu_grad(const float* u, float* out, long long n, void* stream) {
    if (n < 0) return fail(RM_ERR_INVALID_ARG, "n must be >= 0");
    if (n > 0 && (!u || !out)) return fail(RM_ERR_INVALID_ARG, "u / out is NULL");
    RM_CHECK_CUDA(launch_debug_gelu_grad(u, out, n, as_stream(stream)), "debug gelu grad");
    return RM_OK;
}

rm_status rm_moe_pffn_forward_train(rm_ctx* c, int layer, const void* S, float* V_out, float* gates_train,
                                    float* gates_infer, float* lreg, float* A, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (c->cfg.n_experts <= 0) return fail(RM_ERR_UNSUPPORTED, "context was created without experts");
    if (layer < 0 || layer >= c->cfg.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    const LayerW& w = c->layers[layer];
    if (!w.Wg_train) return fail(RM_ERR_UNSUPPORTED, "layer %d has no training router (Wg_train)", layer);
    if ((st = check_batch(c, B)) != RM_OK) return st;
    if (!S || !V_out) return fail(RM_ERR_INVALID_ARG, "S / V_out is NULL");
    if (!aligned16(S) || !aligned16(V_out) || (gates_train && !aligned16(gates_train)) ||
        (gates_infer && !aligned16(gates_infer)))
        return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    cudaSetDevice(c->device);
    cudaStream_t s = as_stream(stream);
    const rm_config& g = c->cfg;
    // the forward on the training router: the layer's experts with h_train's weights in the router slots
    MoeWeights wt = w.moe;
    wt.Wg = w.Wg_train;
    wt.bg = w.bg_train;
    MoeLaunch ml{c->act, S, /*S sample-major*/ true, g.T, g.D, g.n_experts, g.expert_hidden, B, c->Bcap, c->num_sms,
                 c->d_err};
    cudaError_t e = moe_forward(ml, wt, c->moe_ws, V_out, /*V token-major*/ false, gates_train, s,
                                [&](int kind) { return (void*)new ProfScope(c, kind, s); },
                                [](void* p) { delete (ProfScope*)p; });
    if (e != cudaSuccess) return cuda_fail(e, "moe pffn (training router)");
    if (!gates_infer && !lreg && !A) return RM_OK;
    float* gi = gates_infer;
    if (!gi) {
        if (!c->ginfer &&
            (st = dmalloc(c, (void**)&c->ginfer, (size_t)c->Bcap * g.T * g.n_experts * 4, &c->ws_bytes)) != RM_OK)
            return st;
        gi = c->ginfer;
    }
    ProfScope ps(c, RM_K_MOE_ROUTE, s);
    RM_CHECK_CUDA(moe_router_gates(c->act, S, w.moe.Wg, w.moe.bg, gi, B, g.T, g.D, g.n_experts, s),
                  "inference-router gates");
    RM_CHECK_CUDA(moe_gate_sums(gi, lreg, A, B, g.T, g.n_experts, s), "gate sums");
    return RM_OK;
}

rm_status rm_token_mix(const void* X, void* Y, int B, int T, int D, int H, rm_dtype dtype, void* stream) {
    if (!X || !Y) return fail(RM_ERR_INVALID_ARG, "X / Y is NULL");
    if (B < 1 || T < 1 || D < 1 || H < 1) return fail(RM_ERR_INVALID_ARG, "sizes must be positive");
    if (D % H != 0) return fail(RM_ERR_INVALID_ARG, "D (%d) must be divisible by H (%d)", D, H);
    if (dtype != RM_F32 && dtype != RM_BF16) return fail(RM_ERR_INVALID_ARG, "unknown dtype");
    const int esz = dtype == RM_F32 ? 4 : 2;
    const size_t bytes = (size_t)B * T * D * esz;
    const char* x = (const char*)X;
    const char* y = (const char*)Y;
    if (x < y + bytes && y < x + bytes) return fail(RM_ERR_INVALID_ARG, "X and Y overlap");
    RM_CHECK_CUDA(launch_token_mix(X, Y, B, T, D, H, esz, as_stream(stream)), "token mix");
    return RM_OK;
}

rm_status rm_debug_mix_residual(const void* X, int from_z, float* Y, int B, int T, int D, void* stream) {
    if (!X || !Y) return fail(RM_ERR_INVALID_ARG, "X / Y is NULL");
    if (B < 1 || T < 1 || D < 1) return fail(RM_ERR_INVALID_ARG, "sizes must be positive");
    if (D % T != 0) return fail(RM_ERR_INVALID_ARG, "D (%d) must be divisible by T (%d)", D, T);
    if (!aligned16(X) || !aligned16(Y)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    const size_t in_bytes = (size_t)B * T * D * 2, out_bytes = (size_t)B * T * D * 4;
    const char* x = (const char*)X;
    const char* y = (const char*)Y;
    if (x < y + out_bytes && y < x + in_bytes) return fail(RM_ERR_INVALID_ARG, "X and Y overlap");
    int dev = 0, nsm = 0;
    RM_CHECK_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    RM_CHECK_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev), "SM count");
    MixLnArgs a{};
    if (from_z)
        a.Z = X;
    else
        a.X = X;
    a.B = B;
    a.T = T;
    a.D = D;
    a.q = D / T;
    a.Bcap = B;
    a.nchunk = 1;
    a.cw = D;
    a.Ydbg = Y;
    a.timeout_ns = kWaitTimeoutNs;
    cudaError_t e = launch_mix_residual_debug(from_z != 0, a, nsm, as_stream(stream));
    if (e == cudaErrorNotSupported)
        return fail(RM_ERR_UNSUPPORTED, "the staged 8-wide mixing kernel needs D/T %% 8 == 0 and D %% 256 == 0");
    RM_CHECK_CUDA(e, "debug mix residual");
    return RM_OK;
}

rm_status rm_sync_status(rm_ctx* c, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    cudaSetDevice(c->device);
    RM_CHECK_CUDA(cudaStreamSynchronize(as_stream(stream)), "stream synchronize");
    int code = 0;
    RM_CHECK_CUDA(cudaMemcpy(&code, c->d_err, sizeof(int), cudaMemcpyDeviceToHost), "read error word");
    if (code != 0) {
        RM_CHECK_CUDA(cudaMemset(c->d_err, 0, sizeof(int)), "clear error word");
        // a launch that gave up may have left the fused layer's counters part-way: start them again
        if (c->dep_cnt) {
            const size_t ndep = (size_t)c->cfg.T * (size_t)((c->Bcap + 255) / 256);
            RM_CHECK_CUDA(cudaMemset(c->dep_cnt, 0, ndep * sizeof(unsigned)), "clear layer counters");
            c->dep_epoch = 0;
        }
        RM_CHECK_CUDA(cudaDeviceSynchronize(), "clear error word");
        if (code == kDevErrTimeout) return fail(RM_ERR_TIMEOUT, "a device-side wait ran out of time");
        if (code == kDevErrBounds)
            return fail(RM_ERR_DEVICE, "a device-side bounds guard fired (bounds-checked build); the access was skipped");
        return fail(RM_ERR_DEVICE, "device error code %d", code);
    }
    return RM_OK;
}

rm_status rm_get_info(const rm_ctx* c, rm_info* out) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (!out) return fail(RM_ERR_INVALID_ARG, "out is NULL");
    const long long T = c->cfg.T, D = c->cfg.D, k = c->cfg.k, L = c->cfg.L;
    out->params_per_layer = 2 * k * T * D * D + T * (k * D + D) + 4 * D;
    out->flops_per_sample = 4 * k * L * T * D * D;
    out->weight_bytes = c->weight_bytes;
    out->workspace_bytes = c->ws_bytes;
    out->gemm_path = c->use_tc ? RM_PATH_TCGEN05 : RM_PATH_SIMT;
    out->num_sms = c->num_sms;
    out->device = c->device;
    return RM_OK;
}

rm_status rm_profile_enable(rm_ctx* c, int on) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    c->prof = on != 0;
    return RM_OK;
}

rm_status rm_profile_read(rm_ctx* c, rm_kernel_stat* stats) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (!stats) return fail(RM_ERR_INVALID_ARG, "stats is NULL");
    for (int k = 0; k < RM_K_COUNT; ++k) {
        stats[k].launches = 0;
        stats[k].total_ms = 0.0;
    }
    for (auto& u : c->ev_used) {
        Event& e = c->ev_pool[u.second];
        RM_CHECK_CUDA(cudaEventSynchronize(e.b), "event synchronize");
        float ms = 0.f;
        RM_CHECK_CUDA(cudaEventElapsedTime(&ms, e.a, e.b), "event elapsed");
        stats[u.first].launches += 1;
        stats[u.first].total_ms += ms;
    }
    c->ev_used.clear();
    return RM_OK;
}

rm_status rm_debug_gelu(const float* u, float* out, long long n, int form, void* stream) {
    if (n < 0) return fail(RM_ERR_INVALID_ARG, "n must be >= 0");
    if (n > 0 && (!u || !out)) return fail(RM_ERR_INVALID_ARG, "u / out is NULL");
    if (form != 0 && form != 1) return fail(RM_ERR_INVALID_ARG, "form must be 0 (scalar) or 1 (packed)");
    RM_CHECK_CUDA(launch_debug_gelu(u, out, n, form, as_stream(stream)), "debug gelu");
    return RM_OK;
}

rm_status rm_debug_fail_alloc(long long after) {
    AllocBook& b = book();
    std::lock_guard<std::mutex> lk(b.mu);
    b.env_read = true;           // an explicit setting overrides RM_FAULT_INJECT
    b.fail_after = after >= 0 ? after : -1;
    return RM_OK;
}

rm_status rm_debug_alloc_stats(long long* made, long long* live_count, long long* live_bytes) {
    AllocBook& b = book();
    std::lock_guard<std::mutex> lk(b.mu);
    if (made) *made = b.made;
    if (live_count) *live_count = (long long)b.live.size();
    if (live_bytes) *live_bytes = b.live_bytes;
    return RM_OK;
}

rm_status rm_debug_wait_timeout(rm_ctx* c, int timeout_us, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    if (timeout_us < 1 || timeout_us > 10000000) return fail(RM_ERR_INVALID_ARG, "timeout_us out of range");
    cudaSetDevice(c->device);
    RM_CHECK_CUDA(launch_debug_wait(c->d_flag, c->d_err, (unsigned long long)timeout_us * 1000ull, as_stream(stream)),
                  "debug wait");
    return RM_OK;
}

}  // extern "C"

// =============================================================================
// Allocation-free block forward
//
// Some callers cannot allocate device memory at the point where they run the
// model: a serving loop whose memory is owned by a pool or a framework
// allocator that forbids side allocations, a plugin with a fixed memory
// budget, or code that must never trigger the implicit synchronisation a
// cudaMalloc/cudaFree can cause.  rm_block_forward_noalloc serves them: it
// runs the same kernels as rm_block_forward but keeps its intermediates (S,
// the hidden activations, the pre-LN2 rows Z and their row statistics) in
// the file-scope device array below instead of the context's workspace, and
// allocates nothing.  The array is part of the library image, so every GPU
// that loads the library holds it until the process exits.
// =============================================================================
namespace {
constexpr size_t kNoAllocScratchBytes = 32ull << 20;   // 32 MiB
constexpr int kNoAllocMaxDevices = 64;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_base[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on `device` (which must be current).
// The host-side name of the array is not a device address and must never be
// handed to a kernel.  The address is looked up again on every call made
// outside stream capture (the lookup allocates nothing), so a module reloaded
// after a device reset is picked up; under capture the address of the last
// uncaptured call on this device is used.
rm_status noalloc_scratch(int device, cudaStream_t s, void** out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (device < 0 || device >= kNoAllocMaxDevices)
        return fail(RM_ERR_UNSUPPORTED, "allocation-free entry point supports devices 0..%d", kNoAllocMaxDevices - 1);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    RM_CHECK_CUDA(cudaStreamIsCapturing(s, &cap), "cudaStreamIsCapturing");
    if (cap == cudaStreamCaptureStatusNone || !g_noalloc_base[device]) {
        if (cap != cudaStreamCaptureStatusNone)
            return fail(RM_ERR_INVALID_ARG,
                        "the first allocation-free call on a device must come before any stream capture");
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_base[device] = p;
    }
    *out = g_noalloc_base[device];
    return RM_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Layout of the static scratch for B samples (token-major, rows between tokens
// = B): S, Hid and Z in the operand type, the GEMM2 chunk statistics (tensor-
// core path only) and the merged row statistics, each 256-byte aligned.
struct NoAllocLayout {
    size_t S, H, Z, T, R;
    size_t total() const { return S + H + Z + T + R; }
};

NoAllocLayout noalloc_layout(const rm_ctx* c, size_t B) {
    const size_t T = c->cfg.T, D = c->cfg.D, F = c->F, osz = op_size(c->act);
    NoAllocLayout l;
    l.S = align256(T * B * D * osz);
    l.H = align256(T * B * F * osz);
    l.Z = align256(T * B * D * osz);
    l.T = c->use_tc ? align256(T * B * (size_t)c->nchunk * sizeof(float2)) : 0;
    l.R = align256(T * B * sizeof(float2));
    return l;
}

// Largest batch whose intermediates fit the static scratch.
int noalloc_max_batch(const rm_ctx* c) {
    size_t lo = 0, hi = kNoAllocScratchBytes;   // the answer is below hi (every sample takes > 1 byte)
    while (lo < hi) {
        const size_t mid = (lo + hi + 1) / 2;
        if (noalloc_layout(c, mid).total() <= kNoAllocScratchBytes) lo = mid; else hi = mid - 1;
    }
    return lo > (size_t)INT32_MAX ? INT32_MAX : (int)lo;
}

}  // namespace

extern "C" {

rm_status rm_block_forward_noalloc(rm_ctx* c, int layer, const void* X_in, void* X_out, int B, void* stream) {
    rm_status st;
    if ((st = check_ctx(c)) != RM_OK) return st;
    const rm_config& g = c->cfg;
    if (layer < 0 || layer >= g.L) return fail(RM_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (g.moe_layer_mask & (1u << layer))
        return fail(RM_ERR_UNSUPPORTED, "the allocation-free entry point runs dense layers only");
    if (c->layers[layer].um_bs)   // its mixing needs the context's UniMixing workspace
        return fail(RM_ERR_UNSUPPORTED, "the allocation-free entry point runs TokenMixing layers only");
    if (B < 1) return fail(RM_ERR_INVALID_ARG, "B must be >= 1");
    if (!X_in || !X_out) return fail(RM_ERR_INVALID_ARG, "X_in / X_out is NULL");
    if (!aligned16(X_in) || !aligned16(X_out)) return fail(RM_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    const size_t T = g.T, D = g.D, Bs = (size_t)B;
    const size_t io_bytes = Bs * T * D * c->esz;
    const char* xi = (const char*)X_in;
    const char* xo = (const char*)X_out;
    if (xi < xo + io_bytes && xo < xi + io_bytes) return fail(RM_ERR_INVALID_ARG, "X_in and X_out overlap");
    const NoAllocLayout lay = noalloc_layout(c, Bs);
    const size_t need = lay.total();
    if (need > kNoAllocScratchBytes)
        return fail(RM_ERR_INVALID_ARG,
                    "B=%d needs %zu bytes of scratch; the static scratch holds %zu bytes (B <= %d for this "
                    "configuration)",
                    B, need, kNoAllocScratchBytes, noalloc_max_batch(c));
    RM_CHECK_CUDA(cudaSetDevice(c->device), "cudaSetDevice");
    cudaStream_t s = as_stream(stream);
    void* base = nullptr;
    if ((st = noalloc_scratch(c->device, s, &base)) != RM_OK) return st;
    char* p = static_cast<char*>(base);
    void* S = p;
    void* Hid = p + lay.S;
    void* Z = p + lay.S + lay.H;
    float2* stats = reinterpret_cast<float2*>(p + lay.S + lay.H + lay.Z);
    float2* rows = reinterpret_cast<float2*>(p + lay.S + lay.H + lay.Z + lay.T);

    const LayerW& w = c->layers[layer];
    MixLnArgs a = mix_args(c, layer, B);
    a.X = X_in;
    a.S = S;
    a.Bcap = B;
    RM_CHECK_CUDA(launch_mix_ln1(c->act, false, a, c->num_sms, s), "mix+ln1");
    if (c->use_tc) {
        cudaError_t e = launch_gemm1_tc(S, w.W1p, w.b1, Hid, B, g.T, g.D, c->F, B, c->num_sms, c->d_err,
                                        kWaitTimeoutNs, s);
        if (e != cudaSuccess) return cuda_fail(e, (std::string("gemm1 (tcgen05) ") + tc_last_error()).c_str());
        e = launch_gemm2_tc(Hid, w.W2p, w.b2, S, Z, stats, B, g.T, g.D, c->F, B, c->num_sms, c->d_err,
                            kWaitTimeoutNs, s);
        if (e != cudaSuccess) return cuda_fail(e, (std::string("gemm2 (tcgen05) ") + tc_last_error()).c_str());
        RM_CHECK_CUDA(launch_stats_finalize(stats, rows, B, g.T, B, c->nchunk, c->cw, c->num_sms, s),
                      "row statistics");
    } else {
        RM_CHECK_CUDA(launch_gemm1_simt(c->act, S, w.W1p, w.b1, Hid, B, g.T, g.D, c->F, B, s), "gemm1 (simt)");
        RM_CHECK_CUDA(launch_gemm2_simt(c->act, Hid, w.W2p, w.b2, S, Z, B, g.T, g.D, c->F, B, s), "gemm2 (simt)");
        RM_CHECK_CUDA(launch_rowstats(c->act, Z, rows, B, g.T, g.D, B, c->num_sms, s), "row stats");
    }
    RM_CHECK_CUDA(launch_ln2_out(c->act, Z, rows, w.g2, w.be2, X_out, false, B, g.T, g.D, B, 1, g.D, g.ln_eps,
                                 c->num_sms, s),
                  "ln2 out");
    return RM_OK;
}

}  // extern "C"
