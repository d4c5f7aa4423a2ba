/*
 * moe_b300.h -- C ABI of the B300 (sm_103a) forward pass of a token-choice
 * top-k Mixture-of-Experts FFN layer.
 *
 * The layer (pages: "MoE Training: Mixture of Experts", Quick Start
 * MoELayer and Core Concepts; "moe_code.py", MixtureOfExperts.forward;
 * "Mixture of Experts (MoE) From Scratch to DeepSeek V3", routing formula,
 * shared/fine-grained experts, sigmoid routing, aux-loss-free balancing,
 * token dropping; "MoE Training Guide", Core MoE Parameters and Monitoring):
 *
 *   logits = x W_r^T (+ b_r)                                 fp32
 *   keys   = logits (softmax)  |  sigmoid(logits) + b_sel     fp32
 *   top-k experts per token by key, ties to the lower index
 *   gates  = softmax probs | sigmoid scores of the chosen experts,
 *            divided by their sum when renormalize is set
 *   capacity C = max(min_capacity, ceil(T / E * capacity_factor)) when
 *            drop_tokens; slots ranked per expert in priority order (rank j
 *            outer, token inner), rank >= C dropped
 *   per kept slot: y = FFN_e(x_t)  (Linear-GELU-Linear, Linear-ReLU-Linear,
 *            or SwiGLU W2 (silu(W1 x) * W3 x))
 *   out_t  = sum_j gate_tj y_tj + sum_shared FFN_s(x_t) + (residual ? x_t : 0)
 *   stats  = f_e, P_e, L_aux = E sum f_e P_e, z = mean lse^2, drop/imbalance
 *
 * Conventions for every call:
 *   - Pointers are raw device pointers (cudaMalloc'd or torch CUDA tensors)
 *     unless a parameter says "host".  The library never allocates device
 *     memory and never frees a caller's buffer; the caller owns everything.
 *   - Dense tensors are row-major and contiguous.  Weight matrices use the
 *     nn.Linear layout [out_features, in_features]; expert weights are
 *     stacked over experts: w1, w3 [E, d_ff, d_model], w2 [E, d_model, d_ff].
 *   - "dtype" tensors (x, weights, expert biases, out, x_perm) are fp32 or
 *     bf16 as moe_config_t.dtype says.  Router bias, selection bias, logits,
 *     gates, lse, probabilities and y_perm are always fp32.  Index tensors
 *     are int32.
 *   - x, out, x_perm, y_perm and every weight must be 16-byte aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the device.
 *   - Arguments are validated before anything is launched; a failing check
 *     returns a non-zero moe_status_t, launches nothing, and leaves a
 *     message for moe_last_error().  Launch failures return MOE_ERR_CUDA.
 *     A bounded device-side wait that gives up (which only a library bug
 *     or a broken device could cause) sets a device flag read by
 *     moe_check_device_error(); the call then returns without hanging.
 *   - No call throws, aborts or exits.
 *
 * Supported shapes: 1 <= num_experts <= 1024, 1 <= top_k <= min(E, 16),
 * num_tokens >= 0 (0 is a valid empty batch), num_shared in {0, 1}.
 * bf16: d_model and d_ff multiples of 64.  fp32: multiples of 4.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_B300_VERSION 1

typedef void *moe_stream_t; /* cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, bad size      */
    MOE_ERR_UNSUPPORTED = 2,        /* valid layer, shape not supported      */
    MOE_ERR_BAD_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned      */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4,
    MOE_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed  */
    MOE_ERR_DEVICE_TIMEOUT = 6      /* a bounded device-side wait gave up    */
} moe_status_t;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_ACT_GELU = 0, MOE_ACT_RELU = 1, MOE_ACT_SWIGLU = 2 };
enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };

/* Layer description.  Field names follow the DeepSpeed MoE knobs of the
 * "MoE Training Guide" (num_experts, top_k, capacity_factor, min_capacity,
 * drop_tokens). */
typedef struct {
    int64_t num_tokens;    /* T = batch * seq (flattened)                    */
    int32_t d_model;       /* d                                               */
    int32_t num_experts;   /* E routed experts                                */
    int32_t top_k;         /* k                                               */
    int32_t d_ff;          /* F, hidden width of one expert                   */
    int32_t score_fn;      /* MOE_SCORE_*                                     */
    int32_t activation;    /* MOE_ACT_*                                       */
    int32_t dtype;         /* MOE_DTYPE_*: storage of x, weights, out         */
    int32_t renormalize;   /* 1: gates divided by their sum over the top-k    */
    int32_t drop_tokens;   /* 1: apply the capacity limit                     */
    int32_t min_capacity;
    int32_t num_shared;    /* always-on shared experts (0 or 1), weight 1     */
    int32_t residual;      /* 1: out adds x                                   */
    float capacity_factor;
} moe_config_t;

/* Scalars written on the device by moe_stats / moe_forward.  Monitoring
 * metrics of the "MoE Training Guide" (Production Training, Monitoring) and
 * the balance losses of "MoE Training: Mixture of Experts" (Load
 * Balancing). */
typedef struct {
    float aux_loss;        /* E * sum_e f_e P_e (no coefficient applied)      */
    float z_loss;          /* mean_t (logsumexp_e logits_te)^2                */
    float imbalance;       /* max kept_e / min kept_e, +inf if an expert is empty */
    float utilization;     /* #experts with kept_e > 0 / E                    */
    float drop_rate;       /* dropped / (T k)                                 */
    int32_t dropped;       /* sum_e counts_e - kept_e                         */
    int32_t capacity;      /* C, or -1 without token dropping                 */
    int32_t total_kept;    /* sum_e kept_e = rows of x_perm in use            */
} moe_stats_t;

/* Weights of one layer (device pointers).  b_router may be NULL (no router
 * bias).  b1/b2 may be NULL (no expert biases; SwiGLU experts have none).
 * w3 is required for SwiGLU and ignored otherwise.  shared_* are required
 * when num_shared = 1: shared_w1/shared_w3 [F, d], shared_w2 [d, F]. */
typedef struct {
    const void *w_router;  /* [E, d] dtype                                    */
    const float *b_router; /* [E] fp32                                        */
    const void *w1;        /* [E, F, d] dtype                                 */
    const void *b1;        /* [E, F] dtype                                    */
    const void *w3;        /* [E, F, d] dtype                                 */
    const void *w2;        /* [E, d, F] dtype                                 */
    const void *b2;        /* [E, d] dtype                                    */
    const void *shared_w1, *shared_w3, *shared_w2;
} moe_weights_t;

/* Intermediate results of moe_forward.  Each pointer may be NULL, in which
 * case the value is kept in the workspace instead.  Shapes: logits [T,E],
 * topk_idx/topk_w/inv [T*k], lse [T], prob_mean/counts/kept/f [E],
 * offsets [E+1], perm [T*k], stats one moe_stats_t.
 * stage_events: optional host array of MOE_STAGE_EVENTS cudaEvent_t handles
 * (created by the caller) that moe_forward records on its stream at the
 * stage boundaries: [0] start, [1] routed, [2] dispatched, [3] expert
 * first GEMM (W1/W3 + activation) done, [4] expert second GEMM done,
 * [5] shared expert done, [6] combined, [7] statistics done.  NULL: none.
 * Training members (bf16 layers; what moe_backward needs besides the
 * routing members above): x_perm [T*k, d] and hidden [T*k, F] (H, the
 * input of the second expert GEMM) in the layer dtype; pre_act, the first
 * GEMM's pre-activations in bf16: [T*k, 2F] holding W1 x | W3 x for SwiGLU,
 * [T*k, F] holding W1 x + b1 for GELU / ReLU; y_perm [T*k, d] fp32 expert
 * outputs; shared_pre_act [T, 2F or F] and shared_hidden [T, F] for the
 * shared expert.  Rows past offsets[E] are not written. */
#define MOE_STAGE_EVENTS 8
typedef struct {
    float *logits;
    int32_t *topk_idx;
    float *topk_w;
    float *lse;
    float *prob_mean;
    int32_t *counts;
    int32_t *kept;
    int32_t *offsets;
    int32_t *perm;
    int32_t *inv;
    float *f;
    moe_stats_t *stats;
    void *const *stage_events;
    void *x_perm;
    void *pre_act;
    void *hidden;
    float *y_perm;
    void *shared_pre_act;
    void *shared_hidden;
} moe_forward_io_t;

/* Which call a workspace is sized for. */
enum {
    MOE_WS_FORWARD = 0,
    MOE_WS_ROUTE = 1,
    MOE_WS_PERMUTE = 2,
    MOE_WS_EXPERT_FFN = 3,
    MOE_WS_SHARED_FFN = 4,
    MOE_WS_EXPERT_CHOICE = 5,
    MOE_WS_BACKWARD = 6
};

/* Workspace bytes the given call needs (host output).  A workspace sized
 * for MOE_WS_FORWARD is large enough for every call but
 * moe_forward_expert_choice and moe_backward.  Workspace contents
 * need no initialisation and carry nothing between calls. */
moe_status_t moe_workspace_size(const moe_config_t *cfg, int32_t which, size_t *bytes);

/*
 * Router: logits, scores, top-k and gates, with the per-token logsumexp and
 * the balance partials.  Pages: Quick Start MoELayer (gate Linear, softmax,
 * topk, renormalise); DeepSeek V3 page (h(x) = x W_g; sigmoid routing;
 * Score_i = x e_i + b_i used for selection only; fp32 router).
 *   x [T,d] dtype; w_router [E,d] dtype; b_router [E] fp32 or NULL;
 *   sel_bias [E] fp32, required for sigmoid scoring, ignored for softmax.
 * Outputs: logits [T,E] fp32 (bias included); topk_idx [T,k] (descending
 * key, ties to the lower expert index); topk_w [T,k]; lse [T];
 * prob_mean [E] = mean_t softmax(logits_t); counts [E] = slots routed to
 * each expert (before any capacity limit).
 * Workspace: moe_workspace_size(MOE_WS_ROUTE).
 */
moe_status_t moe_route(const moe_config_t *cfg, const void *x, const void *w_router,
                       const float *b_router, const float *sel_bias, float *logits,
                       int32_t *topk_idx, float *topk_w, float *lse, float *prob_mean,
                       int32_t *counts, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Routing from given fp32 logits [T,E] (router bias already included):
 * everything moe_route does after the router GEMM.  Selection is exact on
 * the fp32 keys, so two implementations fed the same logits must agree
 * bit for bit on topk_idx and counts.
 * Workspace: moe_workspace_size(MOE_WS_ROUTE).
 */
moe_status_t moe_route_from_logits(const moe_config_t *cfg, const float *logits,
                                   const float *sel_bias, int32_t *topk_idx, float *topk_w,
                                   float *lse, float *prob_mean, int32_t *counts, void *ws,
                                   size_t ws_bytes, moe_stream_t stream);

/*
 * Dispatch: capacity clamp, stable per-expert ranking in priority order
 * (all rank-0 slots in token order, then rank-1, ...), the permutation and
 * its inverse, and the row copy of x into per-expert contiguous segments.
 * Pages: "MoE Training Guide", Core MoE Parameters (capacity, min capacity,
 * drop_tokens); DeepSeek V3 page, Token Dropping; Quick Start MoELayer
 * masked dispatch x_flat[mask].
 *   topk_idx [T,k] int32, every entry in [0, E) (others are skipped and
 *   flag a device error).
 * Outputs: counts [E]; kept [E] = min(counts, C); offsets [E+1] exclusive
 * prefix of kept; perm [T*k]: perm[row] = slot id t*k+j of that row, -1 for
 * rows >= offsets[E]; inv [T*k]: inv[t*k+j] = row, or -1 if dropped;
 * x_perm [T*k, d] dtype: rows 0 .. offsets[E]-1 written, the rest untouched.
 * Workspace: moe_workspace_size(MOE_WS_PERMUTE).
 */
moe_status_t moe_permute(const moe_config_t *cfg, const void *x, const int32_t *topk_idx,
                         int32_t *counts, int32_t *kept, int32_t *offsets, int32_t *perm,
                         int32_t *inv, void *x_perm, void *ws, size_t ws_bytes,
                         moe_stream_t stream);

/*
 * moe_permute without a workspace, for callers that cannot allocate device
 * memory: code embedded in a host runtime that hands it only its input and
 * output buffers and no allocator (a plugin or custom operator of an
 * inference engine), or that must not allocate after start-up because it
 * runs under a fixed memory budget or latency limit (cudaMalloc and cudaFree
 * can synchronise the device or fail).  The pages have no counterpart; this
 * is a deployment variant of moe_permute.
 *   Same arguments, outputs and results as moe_permute, minus the
 *   workspace.  The two scratch tables live in a 512 KB array of the
 *   library's own device memory (a file-scope __device__ array, present on
 *   every device that loads the library until the process exits).
 *   Limit: ceil(num_tokens * top_k / 2048) * num_experts <= 65536 (for
 *   example T*k <= 16.7M slots at E = 8, <= 524288 at E = 256); larger
 *   layers return MOE_ERR_UNSUPPORTED and must use moe_permute.
 *   The first call on a device looks the array's address up
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  No call allocates or frees device memory.
 *   All calls share the array: every call writes the parts it reads, so
 *   nothing has to be cleared between calls, but calls that overlap on the
 *   GPU (concurrent streams, or several host threads) race on it.
 */
moe_status_t moe_permute_noalloc(const moe_config_t *cfg, const void *x, const int32_t *topk_idx,
                                 int32_t *counts, int32_t *kept, int32_t *offsets, int32_t *perm,
                                 int32_t *inv, void *x_perm, moe_stream_t stream);

/*
 * Routed experts as a grouped GEMM over the segments of x_perm:
 * for rows offsets[e] .. offsets[e+1]-1,
 *   GELU/ReLU: y = W2_e act(W1_e x + b1_e) + b2_e
 *   SwiGLU:    y = W2_e (silu(W1_e x) * (W3_e x))
 * Pages: Quick Start expert nn.Sequential(Linear, GELU, Linear);
 * moe_code.py Expert (ReLU; dropout is the identity in a forward pass);
 * SwiGLU is the three-matrix expert of the Mixtral parameter arithmetic.
 *   x_perm [T*k, d] dtype; offsets [E+1] device; weights as moe_weights_t.
 * Output: y_perm [T*k, d] fp32, rows 0 .. offsets[E]-1 written.
 * The hidden activation H is kept in the workspace in dtype.
 * Workspace: moe_workspace_size(MOE_WS_EXPERT_FFN).
 */
moe_status_t moe_expert_ffn(const moe_config_t *cfg, const void *x_perm, const int32_t *offsets,
                            const void *w1, const void *b1, const void *w3, const void *w2,
                            const void *b2, float *y_perm, void *ws, size_t ws_bytes,
                            moe_stream_t stream);

/*
 * The always-on shared expert (DeepSeek V3 page: shared experts) on every
 * token: z = FFN_shared(x), same activation as the routed experts, no
 * biases.  x [T,d] dtype; shared_w1/w3 [F,d]; shared_w2 [d,F].
 * Output: z [T,d] fp32.  Workspace: moe_workspace_size(MOE_WS_SHARED_FFN).
 */
moe_status_t moe_shared_ffn(const moe_config_t *cfg, const void *x, const void *shared_w1,
                            const void *shared_w3, const void *shared_w2, float *z, void *ws,
                            size_t ws_bytes, moe_stream_t stream);

/*
 * Combine back to token order (Quick Start MoELayer output[mask] +=
 * score * expert_output; DeepSeek V3 page y = sum Gate_i E_i(x) + x):
 *   out_t = sum_{j : inv[t*k+j] >= 0} topk_w[t,j] y_perm[inv[t*k+j]]
 *           + shared_out[t] (if not NULL) + x[t] (if cfg->residual)
 * summed in fp32 in that order (j ascending), stored in dtype.
 *   y_perm [T*k, d] fp32; inv [T*k]; topk_w [T*k]; shared_out [T,d] fp32
 *   or NULL; x [T,d] dtype (required when residual); out [T,d] dtype.
 */
moe_status_t moe_combine(const moe_config_t *cfg, const float *y_perm, const int32_t *inv,
                         const float *topk_w, const float *shared_out, const void *x, void *out,
                         moe_stream_t stream);

/*
 * Balance statistics ("MoE Training: Mixture of Experts", Load Balancing:
 * f_i from bincount of the routed experts over T*k, P_i = mean softmax,
 * aux = N sum f_i P_i, z = mean logsumexp^2; "MoE Training Guide",
 * Monitoring).  counts/kept [E]; prob_mean [E]; lse [T].
 * Outputs: f [E] (may be NULL) and *stats (device).
 */
moe_status_t moe_stats(const moe_config_t *cfg, const int32_t *counts, const int32_t *kept,
                       const float *prob_mean, const float *lse, float *f, moe_stats_t *stats,
                       moe_stream_t stream);

/*
 * Aux-loss-free balancing (DeepSeek V3 page): b_e += gamma * sign(T k / E -
 * counts_e), sign(0) = 0, in place on sel_bias [E] fp32 (device).  counts
 * are the pre-capacity counts of the forward that just ran.
 */
moe_status_t moe_bias_update(const moe_config_t *cfg, const int32_t *counts, float *sel_bias,
                             float gamma, moe_stream_t stream);

/*
 * The whole layer forward: route -> permute -> routed experts (+ shared
 * expert) -> combine -> stats, all on `stream` with no host round trip.
 *   x [T,d] dtype; out [T,d] dtype; io: optional intermediate outputs
 *   (NULL struct or NULL members keep them in the workspace); sel_bias [E]
 *   for sigmoid scoring.  Workspace: moe_workspace_size(MOE_WS_FORWARD).
 */
moe_status_t moe_forward(const moe_config_t *cfg, const moe_weights_t *weights, const void *x,
                         const float *sel_bias, void *out, const moe_forward_io_t *io, void *ws,
                         size_t ws_bytes, moe_stream_t stream);

/*
 * Hash routing ("MoE technical survey" page, Hash layers for large sparse
 * models: a fixed token -> expert mapping, no gating network).  The page
 * gives no hash function; choice j of a token is
 *   fmix32(token_id + j * 0x9E3779B9) mod E
 * (fmix32 = MurmurHash3's 32-bit finalizer), moved to the next expert,
 * cyclically, if an earlier choice of the same token took it; every gate is
 * 1/k.  token_ids [T] int32 (vocabulary ids, any value); outputs
 * topk_idx [T,k] and topk_w [T,k] feed moe_permute / moe_forward_from_routing.
 */
moe_status_t moe_route_hash(const moe_config_t *cfg, const int32_t *token_ids, int32_t *topk_idx,
                            float *topk_w, moe_stream_t stream);

/*
 * The layer forward from routing the caller already has (hash routing, or
 * any other token -> expert assignment): permute -> routed experts (+ shared
 * expert) -> combine -> stats, exactly as moe_forward after its router.
 *   topk_idx [T,k] in [0, E), topk_w [T,k] fp32 (device).  io's routing
 *   members are ignored; stats->aux_loss and z_loss are NaN (no router
 *   probabilities).  Workspace: moe_workspace_size(MOE_WS_FORWARD).
 */
moe_status_t moe_forward_from_routing(const moe_config_t *cfg, const moe_weights_t *weights,
                                      const void *x, const int32_t *topk_idx, const float *topk_w,
                                      void *out, const moe_forward_io_t *io, void *ws,
                                      size_t ws_bytes, moe_stream_t stream);

/*
 * Expert-choice routing ("MoE Training: Mixture of Experts" page, Core
 * Concepts, Routing Mechanisms, Expert Choice Routing): the router's scores
 * are transposed to [experts, tokens] and every expert keeps the C tokens
 * with the largest score, so each expert processes exactly C tokens and a
 * token may be taken by any number of experts, including none.
 *
 * Readings where the page is silent: the score is the router logit
 * (x w_r^T + b_router, fp32); C = min(T, max(min_capacity,
 * ceil(T / E * capacity_factor))) with cfg->capacity_factor (drop_tokens and
 * top_k are not used); equal logits go to the lower token index; the gate
 * of a chosen (token, expert) pair is the token's softmax probability for
 * that expert; a token no expert chose gets only the shared expert and the
 * residual.
 *
 * moe_ec_capacity: host output *capacity = C.
 * moe_route_expert_choice: logits [T,E] fp32 (device, bias included) ->
 *   row_token [E*C] int32: row e*C + i holds the i-th chosen token of
 *   expert e in token order; tok_row [T,E] int32: row of (t, e), -1 if e
 *   did not choose t; tok_gate [T,E] fp32: gate, 0 where not chosen;
 *   offsets [E+1] int32 = e*C.  The selection is exact (no rounding enters
 *   it), so it is reproducible bit for bit from the same logits.
 * Errors: MOE_ERR_INVALID_ARG without a finite capacity_factor > 0;
 *   MOE_ERR_UNSUPPORTED when T * E does not fit in int32.
 */
moe_status_t moe_ec_capacity(const moe_config_t *cfg, int64_t *capacity);
moe_status_t moe_route_expert_choice(const moe_config_t *cfg, const float *logits, int32_t *row_token,
                                     int32_t *tok_row, float *tok_gate, int32_t *offsets,
                                     moe_stream_t stream);

/* Optional outputs of moe_forward_expert_choice (device buffers, sizes as
 * for moe_route_expert_choice; logits [T,E]); NULL members stay in the
 * workspace.  stage_events as in moe_forward_io_t ([1] after routing, [2]
 * after the row gather, [3]/[4] expert GEMMs, [5] shared, [6] = [7]
 * combined: this call computes no balance statistics, as every expert
 * takes exactly C tokens). */
typedef struct {
    float *logits;
    int32_t *row_token;
    int32_t *tok_row;
    float *tok_gate;
    int32_t *offsets;
    void *const *stage_events;
} moe_ec_io_t;

/*
 * The layer forward under expert-choice routing: router logits -> expert
 * choice -> gather of the chosen rows (E*C rows, expert-major) -> routed
 * experts (+ shared expert) -> gate-weighted combine (+ residual), all on
 * `stream`.  x [T,d] and out [T,d] in cfg->dtype.
 * Workspace: moe_workspace_size(MOE_WS_EXPERT_CHOICE) (not covered by
 * MOE_WS_FORWARD).
 */
moe_status_t moe_forward_expert_choice(const moe_config_t *cfg, const moe_weights_t *weights, const void *x,
                                       void *out, const moe_ec_io_t *io, void *ws, size_t ws_bytes,
                                       moe_stream_t stream);

/*
 * Backward of the layer.  No page prints one; the objective is the one the
 * "MoE Training: Mixture of Experts" page trains: the layer output plus the
 * auxiliary load-balancing loss (Load Balancing: loss = main + coef * aux)
 * and the router z-loss,
 *   L = sum_t <dout_t, out_t> + aux_coef * L_aux + z_coef * L_z,
 * (coefficients in opts) differentiated through the forward: gate-weighted combine, expert FFNs
 * (GELU / ReLU / SwiGLU, biases), shared expert, residual, gate function
 * (softmax or sigmoid, renormalised or raw; the selection and the selection
 * bias b_i are piecewise constant and get no gradient), L_aux with the
 * token fractions f_e held fixed, L_z.  Dropped slots pass no gradient.
 *
 * saved: the routing and training members a forward wrote through
 *   moe_forward_io_t (device buffers); counts are the pre-drop counts.
 * x, dout [T, d] bf16.  grads (device, fp32, overwritten): dx [T, d];
 *   dw_router [E, d]; db_router [E] (NULL without router bias); dw1 [E,F,d],
 *   db1 [E,F] (GELU / ReLU with biases), dw3 [E,F,d] (SwiGLU), dw2 [E,d,F],
 *   db2 [E,d]; shared_dw1 / shared_dw3 [F,d], shared_dw2 [d,F].  A NULL
 *   weight gradient is not computed; dx must be given.
 * bf16 layers only (MOE_ERR_UNSUPPORTED for fp32).  The operands the tensor
 * cores consume are stored in bf16 (dy = gate * dout, da); accumulation is
 * fp32.  Workspace: moe_workspace_size(MOE_WS_BACKWARD).
 */
typedef struct {
    const int32_t *topk_idx;
    const float *topk_w;
    const float *logits;
    const int32_t *inv;
    const int32_t *offsets;
    const int32_t *counts;
    const void *x_perm;
    const void *pre_act;
    const void *hidden;
    const float *y_perm;
    const void *shared_pre_act;
    const void *shared_hidden;
} moe_saved_t;

typedef struct {
    float *dx;
    float *dw_router;
    float *db_router;
    float *dw1;
    float *db1;
    float *dw3;
    float *dw2;
    float *db2;
    float *shared_dw1;
    float *shared_dw3;
    float *shared_dw2;
} moe_grads_t;

/* Options of moe_backward (NULL: aux_coef = z_coef = 0, no events).
 * stage_events: optional host array of MOE_BWD_STAGE_EVENTS cudaEvent_t
 * handles recorded on the stream: [0] start, [1] gate and router gradients,
 * [2] dh GEMM with the activation backward, [3] dx GEMM, [4] shared expert
 * data path, [5] dx assembled, [6] dW2 GEMM, [7] dW1 / dW3 GEMMs, [8] bias,
 * router and shared expert weight gradients. */
#define MOE_BWD_STAGE_EVENTS 9
typedef struct {
    float aux_coef;
    float z_coef;
    void *const *stage_events;
} moe_backward_opts_t;

moe_status_t moe_backward(const moe_config_t *cfg, const moe_weights_t *weights, const void *x, const void *dout,
                          const moe_saved_t *saved, const moe_grads_t *grads, const moe_backward_opts_t *opts,
                          void *ws, size_t ws_bytes, moe_stream_t stream);

/* Reads and clears the device error flag (host output *code: 0 = none,
 * else a moe_status_t).  Synchronises the device first. */
moe_status_t moe_check_device_error(int32_t *code);

/*
 * Process-wide switches (all devices, every host thread; they take effect
 * at the next launch).  None is needed in normal use; they exist so that
 * tests can run every kernel variant and exercise the device-side error
 * path without a device fault.
 *   MOE_OPT_PDL            1 (default): the library's kernels are launched
 *                          with programmatic dependent launch; 0: plain
 *                          stream order.
 *   MOE_OPT_GEMM_PAIR      -1 (default): the expert GEMM kernel is chosen by
 *                          shape; 0: always the one-CTA tcgen05 kernel;
 *                          1: the CTA-pair (cta_group::2) kernel wherever
 *                          it takes the problem.
 *   MOE_OPT_WAIT_LIMIT_NS  bound, in ns, of every wait of the GEMM kernels
 *                          on a tensor-core or copy barrier (default 2e9).
 *                          A wait that runs out makes the kernel leave its
 *                          loops, let the copies and MMAs it issued land,
 *                          release its tensor memory and return, and raises
 *                          MOE_ERR_DEVICE_TIMEOUT for moe_check_device_error;
 *                          the outputs of that call are then undefined.
 *                          A limit far below a kernel's run time (a few
 *                          microseconds) forces this path on purpose.
 *   MOE_OPT_GEMM_BAND      -1 (default): an expert GEMM whose experts' rows
 *                          do not fit in L2 walks each expert's tiles in
 *                          bands of M tiles sized from the SM count and the
 *                          operand shapes (N outer, M inner within a band),
 *                          others M fastest over the whole expert; 0: always
 *                          M fastest; n > 0: bands of n M tiles.
 * moe_set_option returns MOE_ERR_INVALID_ARG for an unknown option or a
 * value out of range (PDL 0/1, GEMM_PAIR -1/0/1, WAIT_LIMIT_NS >= 0,
 * GEMM_BAND -1..65536).
 */
enum { MOE_OPT_PDL = 0, MOE_OPT_GEMM_PAIR = 1, MOE_OPT_WAIT_LIMIT_NS = 2, MOE_OPT_GEMM_BAND = 3 };
moe_status_t moe_set_option(int32_t option, int64_t value);
/* Current value of an option (host output). */
moe_status_t moe_get_option(int32_t option, int64_t *value);

/* Message of the last failing call on this host thread (host buffer). */
void moe_last_error(char *buf, size_t len);

/* MOE_B300_VERSION of the built library. */
int32_t moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
