/*
 * rankmixer.h -- C ABI of librankmixer.so, a GB300 (sm_103a) implementation of
 * the RankMixer block forward, its backward (training), the dense-training /
 * sparse-inference MoE forward, and the tokenization and prediction head on
 * either side of the stack.
 *
 * What is computed (per sample, X_n in R^{T x D}, H = T heads of q = D/H):
 *   S_{n-1} = LN1(TokenMixing(X_{n-1}) + X_{n-1})
 *   X_n     = LN2(PFFN(S_{n-1}) + S_{n-1})                      n = 1..L
 *   o       = (1/T) sum_t X_L[t, :]
 * "RankMixer: Scaling Up Ranking Models in Industrial Recommenders", section
 * 3.1 Eq. 1 (block), section 3.3.1 Eq. 3-5 (TokenMixing with H = T), section
 * 3.3.2 Eq. 6-9 (per-token FFN, row-vector convention u = s W + b, GELU),
 * section 3.4 Eq. 10 (ReLU-routed Sparse-MoE variant); "RankMixer 详解（1）"
 * section 3.1 (element map [Mix(X)]_{h, t q + r} = X_{t, h q + r}), section
 * 3.3 (LayerNorm with biased variance, eps inside the square root) and
 * section 4.1 (Gelu(u) = u Phi(u)).
 *
 * Conventions shared by every call:
 *   - Activation tensors are row-major [B][T][D] in the context's dtype
 *     (RM_BF16: __nv_bfloat16 bits, RM_F32: float).  The pooled output and
 *     the MoE PFFN output are always float32.
 *   - Pointers named "device" must be CUDA device (or managed) memory of the
 *     context's device; pointers named "host" must be host memory (pinned for
 *     full copy speed).  Device pointers must be 16-byte aligned.
 *   - "stream" is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Calls taking a stream are asynchronous on it unless
 *     stated otherwise; the caller keeps inputs alive and unmodified until the
 *     stream has passed the call.
 *   - Every call returns an rm_status.  RM_OK means the work was enqueued
 *     (or done, for synchronous calls).  On any other status nothing was
 *     enqueued past the failing launch and rm_last_error() describes why.
 *     No call aborts the process, throws, or prints.
 *   - Errors detected on the device (a bounded wait that ran out) are latched
 *     in a per-context error word and reported by the next rm_sync_status().
 *   - One context may be used by one host thread / one stream at a time; its
 *     workspace is shared by all calls on it.
 *   - The dense forward calls (rm_block_forward, rm_stack_forward, rm_score)
 *     may be captured into a CUDA graph once a first call outside capture has
 *     made the context's lazy allocations: under capture each layer's FFN runs
 *     as two GEMM launches instead of one fused launch (the same results),
 *     because the fused launch depends on per-call host state.
 */
#ifndef RANKMIXER_H_
#define RANKMIXER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RM_ABI_VERSION 4

/* Public symbols are the only ones the shared library exports. */
#if defined(__GNUC__)
#define RM_API __attribute__((visibility("default")))
#else
#define RM_API
#endif

typedef enum rm_status {
    RM_OK = 0,
    RM_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad layer index */
    RM_ERR_UNSUPPORTED = 2,  /* configuration the method or this build does not cover (e.g. H != T) */
    RM_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed; message in rm_last_error() */
    RM_ERR_OOM = 4,          /* device or pinned-host allocation failed */
    RM_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out (reported by rm_sync_status) */
    RM_ERR_DEVICE = 6        /* any other device-side error flag */
} rm_status;

typedef enum rm_dtype {
    RM_F32 = 0,   /* float32 activations and weights, float32 arithmetic */
    RM_BF16 = 1   /* bfloat16 activations and weights, float32 accumulation */
} rm_dtype;

typedef enum rm_gemm_path {
    RM_PATH_AUTO = 0,     /* tcgen05 tensor-core GEMMs when dtype and shape allow, else SIMT */
    RM_PATH_SIMT = 1,     /* CUDA-core GEMMs (any shape, both dtypes) */
    RM_PATH_TCGEN05 = 2   /* require the tcgen05/TMEM path; RM_ERR_UNSUPPORTED if not possible */
} rm_gemm_path;

/* Model shape.  T tokens of width D, H heads (must equal T: the residual in
 * Eq. 5 needs the mixed matrix to keep the [T][D] shape), FFN expansion k
 * (hidden width kD), L stacked blocks.  n_experts > 0 enables the Sparse-MoE
 * PFFN (rm_moe_pffn_forward) with experts of hidden width expert_hidden;
 * moe_layer_mask bit n makes layer n's PFFN the MoE variant inside
 * rm_block_forward / rm_stack_forward.  ln_eps is the LayerNorm epsilon
 * (1e-5 in the pages' worked example).  max_batch bounds B for every call
 * and sizes the context's workspace.  training != 0 makes the context keep a
 * second copy of the dense weights in the pages' layout (bf16 for RM_BF16,
 * float for RM_F32) for rm_block_backward / rm_stack_backward; their
 * workspace is allocated at the first backward call. */
typedef struct rm_config {
    int T;
    int D;
    int H;
    int k;
    int L;
    int n_experts;
    int expert_hidden;
    unsigned moe_layer_mask;
    rm_dtype dtype;
    float ln_eps;
    int max_batch;
    rm_gemm_path gemm_path;
    int training;
} rm_config;

/* Parameters of one layer, as DEVICE pointers in the context's dtype, laid
 * out as the pages write them (row-vector convention, u = s W1 + b1):
 *   W1 [T][D][kD], b1 [T][kD], W2 [T][kD][D], b2 [T][D]    ("RankMixer" Eq. 7)
 *   ln1_gamma, ln1_beta, ln2_gamma, ln2_beta [D]            (one pair per LN,
 *                                                            shared by tokens)
 * Sparse-MoE (only read when n_experts > 0), "RankMixer" Eq. 10:
 *   Wg [T][D][E], bg [T][E]              router h_t(s) = s Wg_t + bg_t, gate ReLU(h)
 *   eW1 [T][E][D][Fe], eb1 [T][E][Fe]    expert first layer (Fe = expert_hidden)
 *   eW2 [T][E][Fe][D], eb2 [T][E][D]     expert second layer
 * Dense-training / sparse-inference MoE ("RankMixer" section 3.4; "6.4
 * Rankmixer: 硬件效率优化" section 6.4.4), optional (NULL: not set):
 *   Wg_train [T][D][E], bg_train [T][E]  the training router h_train; Wg / bg
 *                                        above are h_infer
 * rm_create copies and repacks everything it needs; the caller may free
 * these buffers once rm_create has returned. */
typedef struct rm_layer_params {
    const void *W1, *b1, *W2, *b2;
    const void *ln1_gamma, *ln1_beta, *ln2_gamma, *ln2_beta;
    const void *Wg, *bg;
    const void *eW1, *eb1, *eW2, *eb2;
    const void *Wg_train, *bg_train;
} rm_layer_params;

/* Gradients of one dense layer's parameters, DEVICE float32 buffers in the
 * layout of rm_layer_params ("RankMixer 详解（1）" section 5.2): each is the
 * sum over the batch of the per-sample gradients, and is overwritten.
 *   dW1 [T][D][kD], db1 [T][kD], dW2 [T][kD][D], db2 [T][D],
 *   dln1_gamma, dln1_beta, dln2_gamma, dln2_beta [D]. */
typedef struct rm_layer_grads {
    float *dW1, *db1, *dW2, *db2;
    float *dln1_gamma, *dln1_beta, *dln2_gamma, *dln2_beta;
} rm_layer_grads;

typedef struct rm_ctx rm_ctx;

/* Static facts about a context. */
typedef struct rm_info {
    long long params_per_layer;      /* 2 k T D^2 + biases + LN ("RankMixer" Eq. 12, dense part) */
    long long flops_per_sample;      /* 4 k L T D^2: GEMM flops of the dense stack (Eq. 12) */
    long long weight_bytes;          /* bytes of packed weights held on the device */
    long long workspace_bytes;       /* bytes of activation workspace held on the device */
    int gemm_path;                   /* rm_gemm_path actually used (SIMT or TCGEN05) */
    int num_sms;
    int device;
} rm_info;

/* Kernel classes for rm_profile_read. */
typedef enum rm_kernel_kind {
    RM_K_MIX_LN1 = 0,    /* token mixing + residual + LN1 (and the previous layer's LN2) */
    RM_K_GEMM1 = 1,      /* per-token FFN layer 1 + bias + GELU */
    RM_K_GEMM2 = 2,      /* per-token FFN layer 2 + bias + residual + LN2 row statistics */
    RM_K_LN2_OUT = 3,    /* LN2 finalisation into a [B][T][D] output */
    RM_K_POOL = 4,       /* last LN2 finalisation + mean pooling */
    RM_K_ROWSTATS = 5,   /* LN2 row statistics: (mean, M2) of each full row, merged from the GEMM2 chunk partials */
    RM_K_MOE_ROUTE = 6,  /* router GEMV + ReLU + per-(token, expert) compaction */
    RM_K_MOE_GEMM1 = 7,  /* expert layer 1 + bias + GELU on gathered rows */
    RM_K_MOE_GEMM2 = 8,  /* expert layer 2 + bias, gated, one packed row per (sample, token, open expert) */
    RM_K_MISC = 9,       /* copies, layout changes */
    RM_K_MOE_COMBINE = 10, /* sum of the open experts' gated rows per (sample, token), fixed expert order */
    RM_K_BWD_RECOMPUTE = 11, /* training forward of a layer: LN1 and the per-token FFN keeping S, yhat, Gelu(U), Gelu'(U), Z */
    RM_K_BWD_DGRAD = 12,   /* backward: dA = dZ W2^T (times Gelu'), dS = dU W1^T + dZ */
    RM_K_BWD_WGRAD = 13,   /* backward: dW2 = A^T dZ, dW1 = S^T dU */
    RM_K_BWD_ROWS = 14,    /* backward: LN2 and LN1 + mixing backward, bias / affine reductions */
    RM_K_TOKENIZE = 15,    /* feature tokenization: per-token projection of the embedding slices */
    RM_K_HEAD = 16,        /* prediction head on the pooled output */
    RM_K_UNIMIX = 17,      /* UniMixing: local block products, global product, residual + LN1 */
    RM_K_PFFN = 18,        /* both per-token FFN layers of a dense layer in one launch (B >= 256 on the
                              tensor-core path): the work of RM_K_GEMM1 and RM_K_GEMM2 */
    RM_K_COUNT = 19
} rm_kernel_kind;

typedef struct rm_kernel_stat {
    long long launches;
    double total_ms;
} rm_kernel_stat;

/* ---------------------------------------------------------------------- */

/* Create a context on `device`: validates cfg, allocates workspace for
 * cfg->max_batch samples, repacks the L layers' parameters (layers[0..L-1])
 * into device-resident K-major tiles.  Synchronous.  Errors:
 * RM_ERR_INVALID_ARG (null pointers, non-positive sizes, D % H != 0),
 * RM_ERR_UNSUPPORTED (H != T, or RM_PATH_TCGEN05 requested for a shape or
 * dtype it cannot take), RM_ERR_OOM, RM_ERR_CUDA.  On error *out is NULL. */
RM_API rm_status rm_create(const rm_config *cfg, const rm_layer_params *layers, int device, rm_ctx **out);

/* Release everything the context owns (synchronises its device first). NULL is a no-op. */
RM_API rm_status rm_destroy(rm_ctx *ctx);

/* One block ("RankMixer" Eq. 1) of layer `layer`: X_out = LN2(PFFN(S) + S) with
 * S = LN1(Mix(X_in) + X_in).  X_in: device [B][T][D] in the context dtype.
 * X_out: device [B][T][D] in out_dtype; it may not overlap X_in.  S_out
 * (nullable): device [B][T][D] receives S in out_dtype.  out_dtype is the
 * context dtype or RM_F32: a bf16 context then writes the float32 values
 * that it otherwise rounds to bf16 (round to nearest even), so the two
 * outputs of the same call agree bit for bit after that rounding.  A float32
 * context takes RM_F32 only.  1 <= B <= max_batch.  RM_ERR_INVALID_ARG for
 * another out_dtype. */
RM_API rm_status rm_block_forward(rm_ctx *ctx, int layer, const void *X_in, void *X_out, void *S_out,
                                  rm_dtype out_dtype, int B, void *stream);

/* The whole stack and the mean pooling ("RankMixer" section 3.1): pooled
 * (device float32 [B][D]) = mean_t X_L; XL (nullable, device [B][T][D])
 * receives X_L in xl_dtype (the context dtype, or RM_F32 for the float32
 * values before their rounding, as in rm_block_forward).  X0: device
 * [B][T][D] in the context dtype.  Agrees with chaining rm_block_forward over
 * the layers up to the rounding of each intermediate X_n (the stack keeps them
 * in fp16 on the device, the chained calls round them to their out_dtype). */
RM_API rm_status rm_stack_forward(rm_ctx *ctx, const void *X0, float *pooled, void *XL, rm_dtype xl_dtype, int B,
                                  void *stream);

/* rm_stack_forward from HOST buffers: copies X0_host ([B][T][D], context dtype)
 * to the device, runs the stack, copies the pooled float32 [B][D] result to
 * pooled_host.  Returns after the result is in pooled_host (synchronises the
 * stream).  Uses context-owned device staging buffers.  From B = 2048 on, the
 * batch runs as three chunks, B/8, 3B/8 and the rest (rounded up to multiples
 * of 256 samples), the copy of each chunk overlapping the computation of the
 * previous one (two context-owned copy streams); pinned host buffers let the
 * copies run asynchronously.  Each sample's arithmetic is that of
 * rm_stack_forward. */
RM_API rm_status rm_stack_forward_host(rm_ctx *ctx, const void *X0_host, float *pooled_host, int B, void *stream);

/* Pipelined host entry for a stream of batches (serving): enqueue the stack
 * forward of one batch and return without waiting.  The copy of X0_host
 * ([B][T][D], context dtype) to the device runs on a context-owned copy stream
 * while the previously enqueued batch computes on `stream`; the pooled float32
 * [B][D] result is copied to pooled_host on a second copy stream.  *ticket
 * receives the batch's number; rm_host_wait(ctx, ticket) returns once its
 * pooled_host is written.  Two batches can be in flight (two device staging
 * buffers of max_batch samples, allocated at the first call): a call whose
 * slot still holds the batch two calls back first waits for that batch.  The
 * caller keeps X0_host and pooled_host alive and unmodified until the ticket
 * has been waited for (pinned host memory lets the copies run asynchronously).
 * One batch's arithmetic is that of rm_stack_forward for the same B.
 * rm_host_wait: RM_ERR_INVALID_ARG for a ticket this context never issued;
 * waiting twice, or for a batch that a later call already waited for, returns
 * RM_OK at once. */
RM_API rm_status rm_stack_forward_host_async(rm_ctx *ctx, const void *X0_host, float *pooled_host, int B,
                                             void *stream, long long *ticket);
RM_API rm_status rm_host_wait(rm_ctx *ctx, long long ticket);

/* Sparse-MoE per-token FFN of layer `layer` ("RankMixer" Eq. 10, inference
 * router): V[b,t] = sum_e G[b,t,e] * FFN_{t,e}(S[b,t]) with
 * G = ReLU(S[b,t] Wg_t + bg_t).  Only experts with G > 0 are computed.
 * S: device [B][T][D] (context dtype).  V_out: device float32 [B][T][D].
 * gates (nullable): device float32 [B][T][E] receives G.  Requires
 * cfg.n_experts > 0. */
RM_API rm_status rm_moe_pffn_forward(rm_ctx *ctx, int layer, const void *S, float *V_out, float *gates,
                              int B, void *stream);

/* Training forward of the Sparse-MoE PFFN of layer `layer` with the dense-
 * training / sparse-inference routers ("RankMixer" section 3.4 Eq. 10-11;
 * "6.4 Rankmixer: 硬件效率优化" section 6.4.4):
 *   G_train = ReLU(S Wg_train_t + bg_train_t),  V = sum_e G_train[e] FFN_{t,e}(S)
 *   (the experts with G_train > 0 are computed, as rm_moe_pffn_forward does
 *   for its router), and alongside it
 *   G_infer = ReLU(S Wg_t + bg_t),  lreg[b] = sum_{t,e} G_infer[b][t][e],
 *   A[e] = sum_{b,t} G_infer[b][t][e]  (the regulariser of Eq. 11 per sample,
 *   and each expert's activation over the batch).
 * S: device [B][T][D] (context dtype); V_out: device float32 [B][T][D];
 * gates_train, gates_infer (nullable): device float32 [B][T][E]; lreg
 * (nullable): device float32 [B]; A (nullable): device float32 [E].  Requires
 * cfg.n_experts > 0 and the layer's training router (RM_ERR_UNSUPPORTED
 * otherwise).  Asynchronous on `stream`. */
RM_API rm_status rm_moe_pffn_forward_train(rm_ctx *ctx, int layer, const void *S, float *V_out, float *gates_train,
                                           float *gates_infer, float *lreg, float *A, int B, void *stream);

/* Backward pass of one dense block ("RankMixer 详解（1）" section 5.2) for
 * the loss whose gradient at the block output X' is dX_out:
 *   dZ = LN2 backward of dX_out           (Z = PFFN(S) + S)
 *   dW2 = A^T dZ, db2 = sum dZ, dA = dZ W2^T, dU = dA * Gelu'(U)
 *   dW1 = S^T dU, db1 = sum dU, dS = dU W1^T + dZ
 *   dY = LN1 backward of dS               (Y = Mix(X) + X)
 *   dX_in = dY + P^T dY                   (P the mixing permutation, H = T)
 * The call runs the block's training forward (S, U, Gelu(U), Gelu'(U), Z)
 * from X_in in its own workspace; nothing from an earlier call is needed.
 *   X_in:   device [B][T][D], context dtype (the block's input)
 *   dX_out: device float32 [B][T][D]
 *   dX_in:  device float32 [B][T][D] (may not overlap dX_out)
 *   grads:  host struct of device float32 buffers (see rm_layer_grads);
 *           the sums over the B samples are written, not accumulated.
 * Requires cfg.training != 0 (RM_ERR_UNSUPPORTED otherwise) and a dense layer
 * (RM_ERR_UNSUPPORTED for a Sparse-MoE layer).  bf16 contexts run every
 * product with fp16 operands and float32 accumulation, the gradient operands
 * carrying an exact power-of-two scale per token so that gradients of any
 * magnitude keep fp16's 11 significant bits; float32 contexts run in
 * float32.  The first call allocates the backward workspace for max_batch
 * samples (RM_ERR_OOM if that fails).  Asynchronous on `stream`. */
RM_API rm_status rm_block_backward(rm_ctx *ctx, int layer, const void *X_in, const float *dX_out, float *dX_in,
                                   const rm_layer_grads *grads, int B, void *stream);

/* Training forward of the whole stack: pooled (device float32 [B][D]) = the
 * mean-pooled output of rm_stack_forward, computed by the training kernels
 * (fp16 operands, the same precision as the backward), and every layer's
 * activations that its backward reads (S, the normalised LN1 input and its
 * rstd, Gelu(U), Gelu'(U) and the pre-LN2 rows Z) kept in the context's
 * training workspace for the next rm_stack_backward_saved call.  The first
 * call allocates that workspace: per layer (4 + 2k) x max_batch x T x D
 * half-precision values (float for RM_F32), about 4.4 GB per layer at
 * T = 32, D = 1536, k = 4, max_batch = 4096.  X0: device [B][T][D], context
 * dtype.  Requires cfg.training != 0 and dense layers (RM_ERR_UNSUPPORTED
 * otherwise).  Asynchronous on `stream`. */
RM_API rm_status rm_stack_forward_train(rm_ctx *ctx, const void *X0, float *pooled, int B, void *stream);

/* Backward of the stack and the mean pool from the activations the last
 * rm_stack_forward_train left ("RankMixer 详解（1）" section 5.2), for the
 * loss whose gradient at its pooled output is dpooled (device float32
 * [B][D]): the pool hands each token row dpooled / T, then the layers run
 * backward from the last to the first.  dX0: device float32 [B][T][D];
 * grads: host array of cfg.L structs (layer n at grads[n]), sums over the
 * batch written, not accumulated.  B must be the training forward's batch;
 * the call consumes the saved activations (a second call without a new
 * training forward returns RM_ERR_INVALID_ARG).  Asynchronous on `stream`. */
RM_API rm_status rm_stack_backward_saved(rm_ctx *ctx, const float *dpooled, float *dX0, const rm_layer_grads *grads,
                                         int B, void *stream);

/* rm_stack_forward_train on X0 (into a context-owned pooled buffer) followed by
 * rm_stack_backward_saved: the gradients of the stack for a pooled-output
 * gradient dpooled, from X0 alone.  Same arguments, requirements, workspace
 * and asynchrony as those two calls. */
RM_API rm_status rm_stack_backward(rm_ctx *ctx, const void *X0, const float *dpooled, float *dX0,
                                   const rm_layer_grads *grads, int B, void *stream);

/* Prediction head on the pooled output ("RankMixer 详解（1）" sections 5.1-5.2):
 *   z = pooled[i] . w + b,  p[i] = sigmoid(z),
 *   loss[i] = -y log p - (1 - y) log(1 - p),  dpooled[i] = s (p - y) w,
 * with s = 1 / B when mean_loss (the gradient of the batch-mean loss), else 1.
 * pooled: device float32 [B][D]; w: device float32 [D]; y (nullable): device
 * float32 labels [B]; p, loss (nullable): device float32 [B]; dpooled
 * (nullable): device float32 [B][D].  loss and dpooled need y.  The loss is
 * computed as y softplus(-z) + (1 - y) softplus(z), finite for any z.  Needs
 * no context.  Asynchronous on `stream`. */
RM_API rm_status rm_head_forward(const float *pooled, const float *w, float b, const float *y, float *p,
                                 float *loss, float *dpooled, int B, int D, int mean_loss, void *stream);

/* UniMixing ("UniMixer: A Unified Architecture for Scaling Laws in
 * Recommendation Systems", section 4.3 Eq. 11-15): a learned block-Kronecker
 * mixing in place of a layer's TokenMixing.  Per sample, flatten(X) (L = T D
 * values) is cut into nb = L / bs blocks x_j of bs values and
 *   h_j = x_j WB_j,   out_i = sum_j WG[i][j] h_j,   UniMixing(X) = out_0 | ... | out_{nb-1}
 * with the constrained weights of Eq. 15: each raw matrix W (WG, and every WB_j)
 * is symmetrised, (W + W^T) / 2, divided by the temperature tau and passed to
 * Sinkhorn-Knopp: elementwise exp, then `iters` rounds of dividing every row by
 * its sum and then every column by its sum.  With bs = D / T, WG the block
 * permutation of TokenMixing and WB_j = I it reproduces TokenMixing exactly
 * (the same page, Appendix A).  The layer then runs S = LN1(X + UniMixing(X))
 * and the rest of the block unchanged.
 *
 * rm_set_unimixing: WG device float32 [nb][nb], WB device float32 [nb][bs][bs]
 * (row s, column r of WB_j at WB[j][s][r]), raw (unconstrained); bs must
 * divide T D; tau > 0; iters >= 0; D <= 1536.  Computes the constrained
 * weights on the device (float32, in the log domain: P = exp(C + f_i + g_j)
 * with C = (W + W^T) / (2 tau) and f, g the row and column log-scalings, the
 * same values as the alternating normalisation) and keeps them in the context;
 * the global product runs on fp16 copies in bf16 contexts.  Synchronous: drains
 * `stream` first, returns when done.  Replaces an earlier setting of the layer.
 * Training calls return RM_ERR_UNSUPPORTED on contexts with UniMixing layers.
 * rm_unimixing_weights: copies the constrained weights (device float32, same
 * layouts; either output may be NULL).  rm_unimixing: Y = UniMixing(X) of
 * layer `layer`, X device [B][T][D] in the context dtype, Y device [B][T][D] in
 * out_dtype (the context dtype, or RM_F32 for the values before their bf16
 * rounding).  Asynchronous on `stream`. */
RM_API rm_status rm_set_unimixing(rm_ctx *ctx, int layer, const float *WG, const float *WB, int bs, float tau,
                                  int iters, void *stream);
RM_API rm_status rm_unimixing_weights(rm_ctx *ctx, int layer, float *WG_out, float *WB_out, void *stream);
RM_API rm_status rm_unimixing(rm_ctx *ctx, int layer, const void *X, void *Y, rm_dtype out_dtype, int B,
                              void *stream);

/* Feature tokenization ("RankMixer" section 3.2 Eq. 2; "RankMixer 详解（1）"
 * section 2.4): token t of a sample is the t-th slice of d coordinates of its
 * concatenated embedding, projected to D by token t's own linear layer,
 *   X0[b][t] = E[b][t d : (t + 1) d] W_t + b_t,  W [T][d][D], bias [T][D].
 * rm_set_tokenizer copies W and bias (device, context dtype) into the context
 * (synchronous; replaces an earlier tokenizer).  rm_tokenize: E device
 * [B][T d] in the context dtype -> X0 device [B][T][D] in the context dtype
 * (bf16 contexts: fp16 operands on the tensor cores when d is a multiple of
 * 64 and D of 256, float32 accumulation, one bf16 rounding of X0). */
RM_API rm_status rm_set_tokenizer(rm_ctx *ctx, const void *W, const void *bias, int d);
RM_API rm_status rm_tokenize(rm_ctx *ctx, const void *E, void *X0, int B, void *stream);

/* Backward of rm_tokenize for the gradient dX0 (device float32 [B][T][D]) at
 * its output: dW (device float32 [T][d][D]) = sum_b E_slice^T dX0[b][t],
 * db (device float32 [T][D]) = sum_b dX0[b][t], and, when dE is not NULL,
 * dE (device float32 [B][T d]) slice t = dX0[b][t] W_t^T.  E: the forward's
 * input, device [B][T d] (context dtype).  bf16 contexts run the products on
 * fp16 operands with an exact power-of-two scale per token on dX0.  Sums over
 * the batch are written, not accumulated.  Asynchronous on `stream`. */
RM_API rm_status rm_tokenize_backward(rm_ctx *ctx, const void *E, const float *dX0, float *dE, float *dW, float *db,
                                      int B, void *stream);

/* End-to-end scoring: p[b] = sigmoid(head(pool(stack(tokenize(E[b]))))) with
 * the head's w (device float32 [D]) and b.  E: device [B][T d] (context dtype);
 * p: device float32 [B].  Runs rm_tokenize, rm_stack_forward and
 * rm_head_forward on context-owned buffers (allocated at the first call).
 * Dense stacks only. */
RM_API rm_status rm_score(rm_ctx *ctx, const void *E, const float *head_w, float head_b, float *p, int B,
                          void *stream);

/* Allocation-free variant of rm_block_forward (the paper has no counterpart;
 * this is a deployment aid).  For callers that cannot allocate device memory
 * where they run the model -- a serving loop whose memory belongs to a pool
 * or framework allocator, a plugin with a fixed memory budget, code that must
 * not risk the implicit synchronisation of cudaMalloc/cudaFree.  It computes
 * exactly what rm_block_forward computes for a dense layer, with the same
 * kernels, but keeps the intermediates (S, hidden activations, pre-LN2 rows
 * and their statistics) in one static device array of 32 MiB compiled into
 * the library instead of the context's workspace, and allocates nothing.
 *   - The array exists on every GPU that loads the library until the process
 *     exits.  B is limited by it: a call whose intermediates exceed 32 MiB
 *     returns RM_ERR_INVALID_ARG and names the largest B that fits (on the
 *     tensor-core path B <= 56 at T=32, D=1536, k=4 and B <= 226 at T=16,
 *     D=768, k=4).  B is not limited by cfg.max_batch.
 *   - Each call made outside stream capture looks up the array's device
 *     address on the context's device (a lookup that allocates nothing); a
 *     call under capture reuses the address of the last uncaptured call on
 *     that device.  So make the first call on a device before any stream
 *     capture (a captured first call returns RM_ERR_INVALID_ARG), and after a
 *     device reset make one uncaptured call before capturing again.
 *   - All calls share the array and it keeps the last call's contents.  Every
 *     element a call uses is written earlier in the same call, so nothing
 *     needs clearing, but calls that overlap on the GPU (other streams, other
 *     threads, other contexts) race on it: serialise them.
 *   - Dense TokenMixing layers only (RM_ERR_UNSUPPORTED for a Sparse-MoE
 *     layer, and for a layer set to UniMixing by rm_set_unimixing, whose
 *     mixing uses the context's workspace).
 * X_in, X_out: device [B][T][D] in the context dtype, 16-byte aligned, not
 * overlapping.  Asynchronous on `stream`. */
RM_API rm_status rm_block_forward_noalloc(rm_ctx *ctx, int layer, const void *X_in, void *X_out, int B,
                                          void *stream);

/* Standalone TokenMixing ("RankMixer" Eq. 3-4): Y[b][h][t q + r] = X[b][t][h q + r],
 * q = D / H, for any H dividing D (Y is [B][H][T q]).  A pure permutation of
 * element bits, exact for both dtypes.  X, Y: device, non-overlapping. */
RM_API rm_status rm_token_mix(const void *X, void *Y, int B, int T, int D, int H, rm_dtype dtype, void *stream);

/* Test hook for the mixing inside the fused mix + LN1 kernel ("RankMixer"
 * Eq. 3-5; "RankMixer 详解（1）" section 3.1): runs that kernel's gather and
 * residual sum y[h][t q + r] = X[t][h q + r] + X[h][t q + r] (H = T, q = D/T)
 * and writes y (device float32, token-major [T][B][D]: row h of sample b at
 * (h B + b) D) in place of LN1.
 *   from_z = 0: X is bf16, sample-major [B][T][D] (the first layer's input);
 *               y is the float32 sum of the two gathered values.
 *   from_z = 1: X is fp16, token-major [T][B][D] (the form in which a later
 *               layer's input arrives); the kernel's LN2 finalisation runs as
 *               the identity and y is the fp16 sum (round to nearest even) of
 *               the two gathered values, widened to float32.
 * Needs D % 256 == 0 and (D/T) % 8 == 0 (the shapes the staged kernel
 * serves; RM_ERR_UNSUPPORTED otherwise).  X, Y: device, 16-byte aligned, not
 * overlapping.  Runs on the current device; asynchronous on `stream`. */
RM_API rm_status rm_debug_mix_residual(const void *X, int from_z, float *Y, int B, int T, int D, void *stream);

/* Synchronise `stream`, then report and clear the context's device error
 * word: RM_OK, RM_ERR_TIMEOUT or RM_ERR_DEVICE (or RM_ERR_CUDA if the
 * synchronisation itself failed). */
RM_API rm_status rm_sync_status(rm_ctx *ctx, void *stream);

/* Fill *out with static facts about the context. */
RM_API rm_status rm_get_info(const rm_ctx *ctx, rm_info *out);

/* Per-kernel timing with CUDA events recorded around each launch on the
 * launch stream.  rm_profile_enable(ctx, 1) starts collecting;
 * rm_profile_read synchronises the recorded events, writes RM_K_COUNT
 * entries to stats (launch count and summed milliseconds since the last
 * read) and resets the counters. */
RM_API rm_status rm_profile_enable(rm_ctx *ctx, int on);
RM_API rm_status rm_profile_read(rm_ctx *ctx, rm_kernel_stat *stats);

/* Test hook for failure detection: launches one kernel that waits on a
 * device flag nothing sets, with a bounded wait of timeout_us microseconds;
 * when the wait runs out the kernel latches RM_ERR_TIMEOUT in the context's
 * error word and returns.  The next rm_sync_status() reports it. */
RM_API rm_status rm_debug_wait_timeout(rm_ctx *ctx, int timeout_us, void *stream);

/* Test hooks for allocation failures (host side; no GPU fault is involved).
 * Every device allocation the library makes (context creation and the
 * workspaces its calls allocate on first use) goes through one allocator.
 * rm_debug_fail_alloc(after): with after >= 0, the next `after` allocations
 * succeed and the one after them fails as if the device were out of memory
 * (once; the calling entry point returns RM_ERR_OOM with "injected failure" in
 * rm_last_error()); after < 0 disarms.  RM_FAULT_INJECT=alloc:N in the
 * environment arms the same countdown at the library's first allocation.
 * rm_debug_alloc_stats: allocations made since the library was loaded, and
 * the number and bytes of those still live (any output may be NULL).
 * Process-wide, not per context; thread-safe. */
RM_API rm_status rm_debug_fail_alloc(long long after);
RM_API rm_status rm_debug_alloc_stats(long long *made, long long *live_count, long long *live_bytes);

/* Test hook: out[i] = the GELU the library's GEMM epilogues apply, for n
 * float32 device values (u * Phi(u), "RankMixer 详解（1）" section 4.1, with
 * erf from Abramowitz & Stegun formula 7.1.26, |error in erf| <= 1.5e-7).
 * form 0: the scalar form of the CUDA-core GEMMs; form 1: the packed-pair
 * (fp32x2) form of the tensor-core GEMM epilogues.  Asynchronous on `stream`;
 * RM_ERR_INVALID_ARG for n < 0, NULL buffers or another form. */
RM_API rm_status rm_debug_gelu(const float *u, float *out, long long n, int form, void *stream);

/* Test hook: out[2i] = Gelu(u[i]) and out[2i+1] = Gelu'(u[i]) = Phi(u) + u phi(u)
 * as the backward pass computes them ("RankMixer 详解（1）" section 5.2; Phi by
 * Abramowitz & Stegun 7.1.26).  u: device float32 [n]; out: device float32
 * [2n].  Asynchronous on `stream`; RM_ERR_INVALID_ARG for n < 0 or NULL buffers. */
RM_API rm_status rm_debug_gelu_grad(const float *u, float *out, long long n, void *stream);

/* Message of the last failing call on this host thread ("" if none). */
RM_API const char *rm_last_error(void);

/* ABI version of the loaded library (RM_ABI_VERSION). */
RM_API int rm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RANKMIXER_H_ */
