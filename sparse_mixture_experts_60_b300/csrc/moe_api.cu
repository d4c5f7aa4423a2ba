// C ABI of the MoE-layer forward: argument validation, workspace layout and
// the launch sequence.  Every step of the layer runs in this library's own
// kernels; the host code only checks arguments, carves the caller's
// workspace, encodes TMA descriptors and launches on the caller's stream.
#include <algorithm>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe_b300.h"
#include "moe_internal.h"

using namespace moe;

namespace {

thread_local char g_msg[512] = "";

moe_status_t fail(moe_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

moe_status_t cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MOE_OK;
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int elem_bytes(const moe_config_t *c) { return c->dtype == MOE_DTYPE_F32 ? 4 : 2; }

moe_status_t check_cfg(const moe_config_t *c) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
    if (c->num_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "num_tokens < 0");
    if (c->num_experts < 1 || c->num_experts > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "num_experts must be in [1, %d]", kMaxExperts);
    if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > kMaxTopK)
        return fail(MOE_ERR_INVALID_ARG, "top_k must be in [1, min(num_experts, %d)]", kMaxTopK);
    if (c->d_model < 1 || c->d_ff < 1) return fail(MOE_ERR_INVALID_ARG, "d_model and d_ff must be >= 1");
    if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID)
        return fail(MOE_ERR_INVALID_ARG, "bad score_fn %d", c->score_fn);
    if (c->activation < MOE_ACT_GELU || c->activation > MOE_ACT_SWIGLU)
        return fail(MOE_ERR_INVALID_ARG, "bad activation %d", c->activation);
    if (c->dtype != MOE_DTYPE_F32 && c->dtype != MOE_DTYPE_BF16)
        return fail(MOE_ERR_INVALID_ARG, "bad dtype %d", c->dtype);
    if (c->num_shared != 0 && c->num_shared != 1) return fail(MOE_ERR_UNSUPPORTED, "num_shared must be 0 or 1");
    if (c->drop_tokens && !(c->capacity_factor > 0.0f && isfinite(c->capacity_factor)))
        return fail(MOE_ERR_INVALID_ARG, "capacity_factor must be finite and > 0 with drop_tokens");
    if (c->min_capacity < 0) return fail(MOE_ERR_INVALID_ARG, "min_capacity < 0");
    if (c->num_tokens * (int64_t)c->top_k > INT32_MAX)
        return fail(MOE_ERR_UNSUPPORTED, "num_tokens * top_k must fit in int32");
    if (c->dtype == MOE_DTYPE_BF16 && (c->d_model % 64 || c->d_ff % 64))
        return fail(MOE_ERR_UNSUPPORTED, "bf16 layers need d_model and d_ff multiples of 64");
    if (c->dtype == MOE_DTYPE_F32 && (c->d_model % 4 || c->d_ff % 4))
        return fail(MOE_ERR_UNSUPPORTED, "fp32 layers need d_model and d_ff multiples of 4");
    return MOE_OK;
}

int64_t capacity_of(const moe_config_t *c) {
    const int64_t S = c->num_tokens * c->top_k;
    if (!c->drop_tokens) return S;
    const double v = ceil((double)c->num_tokens / (double)c->num_experts * (double)c->capacity_factor);
    const int64_t cap = (int64_t)v;
    return cap > c->min_capacity ? cap : (int64_t)c->min_capacity;
}

int64_t route_blocks(const moe_config_t *c) { return ceil_div(c->num_tokens, kRouteTokPerCta); }
int64_t perm_chunks(const moe_config_t *c) { return ceil_div(c->num_tokens * c->top_k, kPermChunk); }

// The bf16 router of at most 32 experts runs as one tensor-core GEMM with
// the routing in its epilogue.
bool fused_router(const moe_config_t *c) {
    return c->dtype == MOE_DTYPE_BF16 && c->num_experts <= 32 &&
           grouped_gemm_supported(c->num_experts, c->d_model, 0, 1, 0);
}

size_t route_ws(const moe_config_t *c) {
    return 2 * align256((size_t)route_blocks(c) * c->num_experts * 4) + align256((size_t)route_blocks(c) * 4);
}
// chunk histogram and base tables of the chunked dispatch (the two-launch
// dispatch keeps its chunk table, at most kTwoPassTable entries, in the
// first), and the slots' ranks within their chunk
size_t permute_ws(const moe_config_t *c) {
    const size_t tab = std::max<size_t>((size_t)perm_chunks(c) * c->num_experts, (size_t)kTwoPassTable);
    return 2 * align256(tab * 4) + align256((size_t)c->num_tokens * c->top_k * 4);
}
size_t ffn_ws(const moe_config_t *c) {
    return align256((size_t)c->num_tokens * c->top_k * c->d_ff * elem_bytes(c));
}
size_t shared_ws(const moe_config_t *c) {
    return c->num_shared ? align256((size_t)c->num_tokens * c->d_ff * elem_bytes(c)) : 0;
}

// Bump allocator over the caller's workspace.
struct Carve {
    uint8_t *base;
    size_t used = 0;
    template <typename T>
    T *take(size_t bytes) {
        T *p = reinterpret_cast<T *>(base + used);
        used += align256(bytes);
        return p;
    }
};

size_t forward_ws(const moe_config_t *c) {
    const size_t T = (size_t)c->num_tokens, E = (size_t)c->num_experts, S = T * c->top_k;
    const size_t d = (size_t)c->d_model;
    size_t n = route_ws(c) + permute_ws(c) + ffn_ws(c) + shared_ws(c);
    n += align256(S * d * elem_bytes(c));                         // x_perm
    n += align256(S * d * 4);                                     // y_perm
    if (c->num_shared) n += align256(T * d * 4);                  // z
    n += align256(T * E * 4) + 4 * align256(S * 4) + align256(T * 4);  // logits, idx, w, perm, inv, lse
    n += 4 * align256(E * 4) + align256((E + 1) * 4) + align256(sizeof(moe_stats_t));
    return n;
}

// Expert choice: C = min(T, max(min_capacity, ceil(T / E * capacity_factor))).
int64_t ec_capacity_of(const moe_config_t *c) {
    const int64_t T = c->num_tokens;
    int64_t cap = (int64_t)ceil((double)T / (double)c->num_experts * (double)c->capacity_factor);
    if (cap < c->min_capacity) cap = c->min_capacity;
    return cap < T ? cap : T;
}

size_t ec_ws(const moe_config_t *c) {
    const size_t T = (size_t)c->num_tokens, E = (size_t)c->num_experts, d = (size_t)c->d_model;
    const size_t R = E * (size_t)ec_capacity_of(c), F = (size_t)c->d_ff;
    size_t n = align256(T * E * 4) * 3 + align256(R * 4) + align256((E + 1) * 4);   // logits, tok_row, gate, ...
    n += align256(R * d * elem_bytes(c)) + align256(R * F * elem_bytes(c)) + align256(R * d * 4);
    if (c->num_shared) n += shared_ws(c) + align256(T * d * 4);
    return n;
}

// Backward workspace: R = T k expert rows; the wide router's dlogits and x
// are packed K-major with the T tokens padded to Tp.
struct BwdDims {
    int64_t T, d, E, k, F, nF, R, Rp, Tp;
};
BwdDims bwd_dims(const moe_config_t *c) {
    BwdDims b;
    b.T = c->num_tokens;
    b.d = c->d_model;
    b.E = c->num_experts;
    b.k = c->top_k;
    b.F = c->d_ff;
    b.nF = c->activation == MOE_ACT_SWIGLU ? 2 * b.F : b.F;
    b.R = b.T * b.k;
    b.Rp = (b.R + 64 * b.E + 63) / 64 * 64;
    b.Tp = (b.T + 63) / 64 * 64;
    return b;
}
// Wide routers (E a multiple of 64) take the router's two products with
// the tensor cores (dlogits W_r for dx, dlogits^T x for dW_r).
bool wide_router(const moe_config_t *c) { return c->num_experts >= 64 && c->num_experts % 64 == 0; }

size_t bwd_ws(const moe_config_t *c) {
    const BwdDims b = bwd_dims(c);
    size_t n = align256(b.R * b.d * 2) + align256(b.T * b.k * 4) + align256(b.T * b.E * 4) +
               align256((b.E + 1) * 4) + align256(2 * 4);
    n += align256(b.R * b.nF * 2) + align256(b.R * b.d * 4);                  // da, dx_perm
    n += align256((size_t)router_wgrad_chunks(b.T) * b.E * b.d * 4);
    if (wide_router(c))   // dlogits hi / lo, the router's dx term, [hi | lo]^T, [x^T | x^T]
        n += 2 * align256(b.T * b.E * 2) + align256(b.T * b.d * 4) +
             align256(b.E * 2 * b.Tp * 2) + align256(b.d * 2 * b.Tp * 2) + align256(2 * 4);
    if (c->num_shared) n += align256(b.T * b.nF * 2) + align256(b.T * b.d * 4);
    return n;
}

// ------------------------------------------------------------------ step bodies (no validation)
// logits [T,E] = x w_r^T + b_router (tensor cores for bf16 where the GEMM takes the shape)
moe_status_t router_logits_impl(const moe_config_t *c, const void *x, const void *w_router, const float *b_router,
                                float *logits, cudaStream_t s) {
    if (c->num_tokens == 0) return MOE_OK;
    cudaError_t e;
    if (c->dtype == MOE_DTYPE_BF16 && grouped_gemm_supported(c->num_experts, c->d_model, 0, 1, 0)) {
        GemmProblem g{};
        g.A = static_cast<const bf16 *>(x);
        g.a_rows = c->num_tokens;
        g.B = static_cast<const bf16 *>(w_router);
        g.b_rows_total = c->num_experts;
        g.b_group_rows = c->num_experts;
        g.G = 1;
        g.M = (int)c->num_tokens;
        g.N = c->num_experts;
        g.K = c->d_model;
        g.out = logits;
        g.ldo = c->num_experts;
        g.out_f32 = 1;
        e = launch_grouped_gemm(g, s);
    } else {
        RouteParams p{};
        p.T = c->num_tokens;
        p.E = c->num_experts;
        p.d = c->d_model;
        p.x = x;
        p.w_router = w_router;
        p.logits = logits;
        e = launch_router_logits_simt(p, c->dtype, s);
    }
    if (e == cudaSuccess) e = launch_add_bias(logits, b_router, c->num_tokens, c->num_experts, s);
    return cuda_status(e, "router logits launch");
}

moe_status_t ec_route_impl(const moe_config_t *c, const float *logits, int32_t *row_token, int32_t *tok_row,
                           float *tok_gate, int32_t *offsets, cudaStream_t s) {
    cudaError_t e = launch_ec_select(logits, c->num_tokens, c->num_experts, ec_capacity_of(c), row_token, tok_row,
                                     offsets, s);
    if (e == cudaSuccess) e = launch_ec_gates(logits, tok_row, c->num_tokens, c->num_experts, tok_gate, s);
    return cuda_status(e, "expert-choice routing launch");
}

// Per-32-token routing partials in the route workspace.
struct RoutePartials {
    float *prob;       // [E, nblk]
    int32_t *cnt;      // [E, nblk]
    float *z;          // [nblk]
    int64_t nblk;
};
RoutePartials route_partials(const moe_config_t *c, void *ws) {
    Carve cv{static_cast<uint8_t *>(ws)};
    RoutePartials r;
    r.nblk = route_blocks(c);
    r.prob = cv.take<float>((size_t)r.nblk * c->num_experts * 4);
    r.cnt = cv.take<int32_t>((size_t)r.nblk * c->num_experts * 4);
    r.z = cv.take<float>((size_t)r.nblk * 4);
    return r;
}

// reduce = false (the layer forward): prob_mean / counts are not reduced
// here; the statistics kernel reads the partials.
moe_status_t route_impl(const moe_config_t *c, const void *x, const void *w_router, const float *b_router,
                        const float *sel_bias, float *logits, const float *logits_in, int32_t *topk_idx,
                        float *topk_w, float *lse, float *prob_mean, int32_t *counts, void *ws,
                        cudaStream_t s, bool reduce = true) {
    const RoutePartials rp = route_partials(c, ws);
    const int64_t nblk = rp.nblk;
    float *part_prob = rp.prob;
    int32_t *part_cnt = rp.cnt;
    RouteParams p{};
    p.T = c->num_tokens;
    p.E = c->num_experts;
    p.k = c->top_k;
    p.d = c->d_model;
    p.score_fn = c->score_fn;
    p.renormalize = c->renormalize;
    p.x = x;
    p.w_router = w_router;
    p.b_router = b_router;
    p.sel_bias = sel_bias;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.lse = lse;
    p.part_prob = part_prob;
    p.part_cnt = part_cnt;
    p.part_z = rp.z;
    cudaError_t e = cudaSuccess;
    const bool fused_gemm = !logits_in && fused_router(c);
    if (fused_gemm) {
        // bf16, E <= 32: logits on the tensor cores with the routing in the
        // GEMM's epilogue (one launch)
        if (c->num_tokens > 0) {
            RouteEpilogue re{};
            re.b_router = b_router;
            re.sel_bias = sel_bias;
            re.k = c->top_k;
            re.score_fn = c->score_fn;
            re.renormalize = c->renormalize;
            re.topk_idx = topk_idx;
            re.topk_w = topk_w;
            re.lse = lse;
            re.part_prob = part_prob;
            re.part_cnt = part_cnt;
            re.part_z = rp.z;
            re.nblk = nblk;
            GemmProblem g{};
            g.A = static_cast<const bf16 *>(x);
            g.a_rows = c->num_tokens;
            g.B = static_cast<const bf16 *>(w_router);
            g.b_rows_total = c->num_experts;
            g.b_group_rows = c->num_experts;
            g.G = 1;
            g.M = (int)c->num_tokens;
            g.N = c->num_experts;
            g.K = c->d_model;
            g.out = logits;
            g.ldo = c->num_experts;
            g.out_f32 = 1;
            g.route = &re;
            e = launch_grouped_gemm(g, s);
        }
    } else if (logits_in) {
        p.logits = const_cast<float *>(logits_in);
        p.logits_add_bias = 0;
        e = launch_route_logits(p, s);
    } else if (c->dtype == MOE_DTYPE_F32 && c->num_experts <= 32) {
        p.logits = logits;
        e = launch_router_fused(p, s);
    } else {
        // bf16: logits on the tensor cores (x streamed once by TMA), then the
        // routing kernel adds the router bias and selects
        p.logits = logits;
        p.logits_add_bias = 1;
        if (c->num_tokens > 0) {
            if (c->dtype == MOE_DTYPE_BF16 && grouped_gemm_supported(c->num_experts, c->d_model, 0, 1, 0)) {
                GemmProblem g{};
                g.A = static_cast<const bf16 *>(x);
                g.a_rows = c->num_tokens;
                g.B = static_cast<const bf16 *>(w_router);
                g.b_rows_total = c->num_experts;
                g.b_group_rows = c->num_experts;
                g.seg = nullptr;
                g.G = 1;
                g.M = (int)c->num_tokens;
                g.N = c->num_experts;
                g.K = c->d_model;
                g.out = logits;
                g.ldo = c->num_experts;
                g.out_f32 = 1;
                e = launch_grouped_gemm(g, s);
            } else {
                e = launch_router_logits_simt(p, c->dtype, s);
            }
        }
        if (e == cudaSuccess) e = launch_route_logits(p, s);
    }
    if (e == cudaSuccess && reduce)
        e = launch_route_reduce(part_prob, part_cnt, nblk, c->num_experts, c->num_tokens, prob_mean, counts, s);
    return cuda_status(e, "moe_route launch");
}

moe_status_t permute_impl(const moe_config_t *c, const void *x, const int32_t *topk_idx, int32_t *counts,
                          int32_t *kept, int32_t *offsets, int32_t *perm, int32_t *inv, void *x_perm,
                          void *ws, cudaStream_t s) {
    Carve cv{static_cast<uint8_t *>(ws)};
    const int64_t nch = perm_chunks(c);
    PermuteParams p{};
    p.T = c->num_tokens;
    p.E = c->num_experts;
    p.k = c->top_k;
    p.d = c->d_model;
    p.dtype = c->dtype;
    p.cap = capacity_of(c);
    p.x = x;
    p.topk_idx = topk_idx;
    p.counts = counts;
    p.kept = kept;
    p.offsets = offsets;
    p.perm = perm;
    p.inv = inv;
    p.x_perm = x_perm;
    const size_t tab = std::max<size_t>((size_t)nch * c->num_experts, (size_t)kTwoPassTable);
    p.hist = cv.take<int32_t>(tab * 4);
    p.base = cv.take<int32_t>(tab * 4);
    p.lrank = cv.take<int32_t>((size_t)c->num_tokens * c->top_k * 4);
    return cuda_status(launch_permute(p, s), "moe_permute launch");
}

// Two-layer FFN over row groups (routed: seg = offsets, G = E; shared: seg = null).
moe_status_t ffn_impl(const moe_config_t *c, const void *A, int64_t a_rows, const int32_t *seg, int G, int M,
                      const void *w1, const void *b1, const void *w3, const void *w2, const void *b2, void *H,
                      float *y, cudaStream_t s, void *mid_event = nullptr, void *pre = nullptr,
                      const CombinePrep *comb = nullptr) {
    const int d = c->d_model, F = c->d_ff;
    const int gated = c->activation == MOE_ACT_SWIGLU;
    const int act = c->activation == MOE_ACT_GELU ? 1 : (c->activation == MOE_ACT_RELU ? 2 : 0);
    if (a_rows == 0) return MOE_OK;
    cudaError_t e;
    if (c->dtype == MOE_DTYPE_BF16) {
        GemmProblem g1{};
        g1.A = static_cast<const bf16 *>(A);
        g1.a_rows = a_rows;
        g1.B = static_cast<const bf16 *>(w1);
        g1.B2 = static_cast<const bf16 *>(w3);
        g1.b_rows_total = (int64_t)G * F;
        g1.b_group_rows = F;
        g1.seg = seg;
        g1.G = G;
        g1.M = M;
        g1.N = F;
        g1.K = d;
        g1.out = H;
        g1.ldo = F;
        g1.out_f32 = 0;
        g1.bias = gated ? nullptr : static_cast<const bf16 *>(b1);
        g1.bias_stride = F;
        g1.act = act;
        g1.gated = gated;
        g1.pre = static_cast<bf16 *>(pre);
        g1.ld_pre = gated ? 2 * (int64_t)F : F;
        e = launch_grouped_gemm(g1, s);
        if (e != cudaSuccess) return cuda_status(e, "expert FFN1 launch");
        if (mid_event) cudaEventRecord(static_cast<cudaEvent_t>(mid_event), s);
        GemmProblem g2{};
        g2.A = static_cast<const bf16 *>(H);
        g2.a_rows = a_rows;
        g2.B = static_cast<const bf16 *>(w2);
        g2.b_rows_total = (int64_t)G * d;
        g2.b_group_rows = d;
        g2.seg = seg;
        g2.G = G;
        g2.M = M;
        g2.N = d;
        g2.K = F;
        g2.out = y;
        g2.ldo = d;
        g2.out_f32 = 1;
        g2.bias = gated ? nullptr : static_cast<const bf16 *>(b2);
        g2.bias_stride = d;
        g2.act = 0;
        g2.gated = 0;
        if (comb) g2.comb = *comb;
        e = launch_grouped_gemm(g2, s);
        return cuda_status(e, "expert FFN2 launch");
    }
    if (pre) return fail(MOE_ERR_UNSUPPORTED, "training members (pre-activations) need a bf16 layer");
    SimtProblem p1{};
    p1.A = static_cast<const float *>(A);
    p1.B = static_cast<const float *>(w1);
    p1.B2 = static_cast<const float *>(w3);
    p1.seg = seg;
    p1.G = G;
    p1.M = M;
    p1.max_rows = a_rows;
    p1.N = F;
    p1.K = d;
    p1.out = static_cast<float *>(H);
    p1.ldo = F;
    p1.bias = gated ? nullptr : static_cast<const float *>(b1);
    p1.bias_stride = F;
    p1.act = act;
    p1.gated = gated;
    e = launch_ffn_simt(p1, s);
    if (e != cudaSuccess) return cuda_status(e, "expert FFN1 launch");
    if (mid_event) cudaEventRecord(static_cast<cudaEvent_t>(mid_event), s);
    SimtProblem p2{};
    p2.A = static_cast<const float *>(H);
    p2.B = static_cast<const float *>(w2);
    p2.seg = seg;
    p2.G = G;
    p2.M = M;
    p2.max_rows = a_rows;
    p2.N = d;
    p2.K = F;
    p2.out = y;
    p2.ldo = d;
    p2.bias = gated ? nullptr : static_cast<const float *>(b2);
    p2.bias_stride = d;
    p2.act = 0;
    p2.gated = 0;
    return cuda_status(launch_ffn_simt(p2, s), "expert FFN2 launch");
}

// A buffer of n > 0 elements must be non-NULL (16-byte aligned for need16);
// an empty buffer (n == 0) may be NULL.
moe_status_t need(const void *p, const char *name, int64_t n = 1) {
    if (n == 0) return MOE_OK;
    return p ? MOE_OK : fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
}
moe_status_t need16(const void *p, const char *name, int64_t n = 1) {
    if (n == 0 && !p) return MOE_OK;
    if (!p) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
    return aligned16(p) ? MOE_OK : fail(MOE_ERR_BAD_ALIGNMENT, "%s is not 16-byte aligned", name);
}
moe_status_t need_ws(const void *ws, size_t have, size_t want) {
    if (want == 0) return MOE_OK;
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL (%zu bytes needed)", want);
    if (have < want) return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, %zu needed", have, want);
    if (!aligned16(ws)) return fail(MOE_ERR_BAD_ALIGNMENT, "workspace is not 16-byte aligned");
    return MOE_OK;
}

#define TRY(x)                             \
    do {                                   \
        moe_status_t st_ = (x);            \
        if (st_ != MOE_OK) return st_;     \
    } while (0)

moe_status_t check_weights_ffn(const moe_config_t *c, const void *w1, const void *w3, const void *w2) {
    TRY(need16(w1, "w1"));
    TRY(need16(w2, "w2"));
    if (c->activation == MOE_ACT_SWIGLU) TRY(need16(w3, "w3 (SwiGLU)"));
    return MOE_OK;
}
moe_status_t check_bias(const void *b) {
    return (b && !aligned16(b)) ? fail(MOE_ERR_BAD_ALIGNMENT, "expert bias is not 16-byte aligned") : MOE_OK;
}

moe_status_t check_ec(const moe_config_t *c) {
    if (!(c->capacity_factor > 0.0f && isfinite(c->capacity_factor)))
        return fail(MOE_ERR_INVALID_ARG, "expert choice needs a finite capacity_factor > 0");
    if (c->num_tokens * (int64_t)c->num_experts > INT32_MAX)
        return fail(MOE_ERR_UNSUPPORTED, "expert choice needs num_tokens * num_experts to fit in int32");
    return MOE_OK;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

int32_t moe_version(void) { return MOE_B300_VERSION; }

void moe_last_error(char *buf, size_t len) {
    if (!buf || len == 0) return;
    snprintf(buf, len, "%s", g_msg);
}

moe_status_t moe_workspace_size(const moe_config_t *cfg, int32_t which, size_t *bytes) {
    TRY(check_cfg(cfg));
    TRY(need(bytes, "bytes"));
    switch (which) {
        case MOE_WS_FORWARD: *bytes = forward_ws(cfg); return MOE_OK;
        case MOE_WS_ROUTE: *bytes = route_ws(cfg); return MOE_OK;
        case MOE_WS_PERMUTE: *bytes = permute_ws(cfg); return MOE_OK;
        case MOE_WS_EXPERT_FFN: *bytes = ffn_ws(cfg); return MOE_OK;
        case MOE_WS_SHARED_FFN: *bytes = shared_ws(cfg); return MOE_OK;
        case MOE_WS_EXPERT_CHOICE: TRY(check_ec(cfg)); *bytes = ec_ws(cfg); return MOE_OK;
        case MOE_WS_BACKWARD: *bytes = bwd_ws(cfg); return MOE_OK;
        default: return fail(MOE_ERR_INVALID_ARG, "unknown workspace kind %d", which);
    }
}

moe_status_t moe_route(const moe_config_t *cfg, const void *x, const void *w_router, const float *b_router,
                       const float *sel_bias, float *logits, int32_t *topk_idx, float *topk_w, float *lse,
                       float *prob_mean, int32_t *counts, void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    TRY(need16(x, "x", T));
    TRY(need16(w_router, "w_router"));
    TRY(need(logits, "logits", T));
    TRY(need(topk_idx, "topk_idx", S));
    TRY(need(topk_w, "topk_w", S));
    TRY(need(lse, "lse", T));
    TRY(need(prob_mean, "prob_mean"));
    TRY(need(counts, "counts"));
    if (cfg->score_fn == MOE_SCORE_SIGMOID) TRY(need(sel_bias, "sel_bias (sigmoid scoring)"));
    TRY(need_ws(ws, ws_bytes, route_ws(cfg)));
    return route_impl(cfg, x, w_router, b_router, cfg->score_fn == MOE_SCORE_SIGMOID ? sel_bias : nullptr,
                      logits, nullptr, topk_idx, topk_w, lse, prob_mean, counts, ws,
                      static_cast<cudaStream_t>(stream));
}

moe_status_t moe_route_from_logits(const moe_config_t *cfg, const float *logits, const float *sel_bias,
                                   int32_t *topk_idx, float *topk_w, float *lse, float *prob_mean,
                                   int32_t *counts, void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    TRY(need(logits, "logits", T));
    TRY(need(topk_idx, "topk_idx", S));
    TRY(need(topk_w, "topk_w", S));
    TRY(need(lse, "lse", T));
    TRY(need(prob_mean, "prob_mean"));
    TRY(need(counts, "counts"));
    if (cfg->score_fn == MOE_SCORE_SIGMOID) TRY(need(sel_bias, "sel_bias (sigmoid scoring)"));
    TRY(need_ws(ws, ws_bytes, route_ws(cfg)));
    return route_impl(cfg, nullptr, nullptr, nullptr, cfg->score_fn == MOE_SCORE_SIGMOID ? sel_bias : nullptr,
                      nullptr, logits, topk_idx, topk_w, lse, prob_mean, counts, ws,
                      static_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute(const moe_config_t *cfg, const void *x, const int32_t *topk_idx, int32_t *counts,
                         int32_t *kept, int32_t *offsets, int32_t *perm, int32_t *inv, void *x_perm, void *ws,
                         size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    TRY(need16(x, "x", T));
    TRY(need(topk_idx, "topk_idx", S));
    TRY(need(counts, "counts"));
    TRY(need(kept, "kept"));
    TRY(need(offsets, "offsets"));
    TRY(need(perm, "perm", S));
    TRY(need(inv, "inv", S));
    TRY(need16(x_perm, "x_perm", S));
    TRY(need_ws(ws, ws_bytes, permute_ws(cfg)));
    return permute_impl(cfg, x, topk_idx, counts, kept, offsets, perm, inv, x_perm, ws,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute_noalloc(const moe_config_t *cfg, const void *x, const int32_t *topk_idx, int32_t *counts,
                                 int32_t *kept, int32_t *offsets, int32_t *perm, int32_t *inv, void *x_perm,
                                 moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    TRY(need16(x, "x", T));
    TRY(need(topk_idx, "topk_idx", S));
    TRY(need(counts, "counts"));
    TRY(need(kept, "kept"));
    TRY(need(offsets, "offsets"));
    TRY(need(perm, "perm", S));
    TRY(need(inv, "inv", S));
    TRY(need16(x_perm, "x_perm", S));
    const int64_t table = perm_chunks(cfg) * cfg->num_experts;
    if (2 * table > kPermStaticScratchInts)
        return fail(MOE_ERR_UNSUPPORTED,
                    "moe_permute_noalloc: ceil(num_tokens*top_k/%d) * num_experts = %lld exceeds the static "
                    "scratch limit of %lld; use moe_permute with a workspace",
                    kPermChunk, (long long)table, (long long)(kPermStaticScratchInts / 2));
    int32_t *scratch = permute_static_scratch();
    if (!scratch) return fail(MOE_ERR_CUDA, "moe_permute_noalloc: cudaGetSymbolAddress of the scratch failed");
    PermuteParams p{};
    p.T = T;
    p.E = cfg->num_experts;
    p.k = cfg->top_k;
    p.d = cfg->d_model;
    p.dtype = cfg->dtype;
    p.cap = capacity_of(cfg);
    p.x = x;
    p.topk_idx = topk_idx;
    p.counts = counts;
    p.kept = kept;
    p.offsets = offsets;
    p.perm = perm;
    p.inv = inv;
    p.x_perm = x_perm;
    p.hist = scratch;
    p.base = scratch + table;
    p.chunked = 1;
    return cuda_status(launch_permute(p, static_cast<cudaStream_t>(stream)), "moe_permute_noalloc launch");
}

moe_status_t moe_expert_ffn(const moe_config_t *cfg, const void *x_perm, const int32_t *offsets, const void *w1,
                            const void *b1, const void *w3, const void *w2, const void *b2, float *y_perm,
                            void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t S = cfg->num_tokens * cfg->top_k;
    TRY(need16(x_perm, "x_perm", S));
    TRY(need(offsets, "offsets"));
    TRY(check_weights_ffn(cfg, w1, w3, w2));
    TRY(check_bias(b1));
    TRY(check_bias(b2));
    TRY(need16(y_perm, "y_perm", S));
    TRY(need_ws(ws, ws_bytes, ffn_ws(cfg)));
    return ffn_impl(cfg, x_perm, cfg->num_tokens * cfg->top_k, offsets, cfg->num_experts, 0, w1, b1, w3, w2, b2,
                    ws, y_perm, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_shared_ffn(const moe_config_t *cfg, const void *x, const void *shared_w1, const void *shared_w3,
                            const void *shared_w2, float *z, void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    if (cfg->num_shared != 1) return fail(MOE_ERR_INVALID_ARG, "moe_shared_ffn needs num_shared = 1");
    TRY(need16(x, "x", cfg->num_tokens));
    TRY(check_weights_ffn(cfg, shared_w1, shared_w3, shared_w2));
    TRY(need16(z, "z", cfg->num_tokens));
    TRY(need_ws(ws, ws_bytes, shared_ws(cfg)));
    return ffn_impl(cfg, x, cfg->num_tokens, nullptr, 1, (int)cfg->num_tokens, shared_w1, nullptr, shared_w3,
                    shared_w2, nullptr, ws, z, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const moe_config_t *cfg, const float *y_perm, const int32_t *inv, const float *topk_w,
                         const float *shared_out, const void *x, void *out, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    TRY(need16(y_perm, "y_perm", S));
    TRY(need(inv, "inv", S));
    TRY(need(topk_w, "topk_w", S));
    if (shared_out) TRY(need16(shared_out, "shared_out"));
    if (cfg->residual) TRY(need16(x, "x (residual)", T));
    TRY(need16(out, "out", T));
    return cuda_status(launch_combine(cfg->num_tokens, cfg->d_model, cfg->top_k, cfg->dtype, y_perm, inv, topk_w,
                                      shared_out, cfg->residual ? x : nullptr, out,
                                      static_cast<cudaStream_t>(stream)),
                       "moe_combine launch");
}

moe_status_t moe_stats(const moe_config_t *cfg, const int32_t *counts, const int32_t *kept, const float *prob_mean,
                       const float *lse, float *f, moe_stats_t *stats, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    TRY(need(counts, "counts"));
    TRY(need(kept, "kept"));
    TRY(need(prob_mean, "prob_mean"));
    if (cfg->num_tokens > 0) TRY(need(lse, "lse"));
    TRY(need(stats, "stats"));
    StatsParams p{};
    p.T = cfg->num_tokens;
    p.E = cfg->num_experts;
    p.k = cfg->top_k;
    p.cap = capacity_of(cfg);
    p.drop = cfg->drop_tokens;
    p.counts = counts;
    p.kept = kept;
    p.prob_mean = prob_mean;
    p.lse = lse;
    p.f = f;
    p.stats = stats;
    return cuda_status(launch_stats(p, static_cast<cudaStream_t>(stream)), "moe_stats launch");
}

moe_status_t moe_bias_update(const moe_config_t *cfg, const int32_t *counts, float *sel_bias, float gamma,
                             moe_stream_t stream) {
    TRY(check_cfg(cfg));
    TRY(need(counts, "counts"));
    TRY(need(sel_bias, "sel_bias"));
    if (!isfinite(gamma)) return fail(MOE_ERR_INVALID_ARG, "gamma must be finite");
    return cuda_status(launch_bias_update(cfg->num_tokens, cfg->num_experts, cfg->top_k, counts, sel_bias, gamma,
                                          static_cast<cudaStream_t>(stream)),
                       "moe_bias_update launch");
}

}  // extern "C"

namespace {
moe_status_t forward_impl(const moe_config_t *cfg, const moe_weights_t *w, const void *x, const float *sel_bias,
                          const int32_t *given_idx, const float *given_w, void *out, const moe_forward_io_t *io,
                          void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    TRY(need(w, "weights"));
    TRY(need16(x, "x", cfg->num_tokens));
    TRY(need16(out, "out", cfg->num_tokens));
    if (!given_idx) TRY(need16(w->w_router, "w_router"));
    TRY(check_weights_ffn(cfg, w->w1, w->w3, w->w2));
    TRY(check_bias(w->b1));
    TRY(check_bias(w->b2));
    if (cfg->num_shared) TRY(check_weights_ffn(cfg, w->shared_w1, w->shared_w3, w->shared_w2));
    if (!given_idx && cfg->score_fn == MOE_SCORE_SIGMOID) TRY(need(sel_bias, "sel_bias (sigmoid scoring)"));
    TRY(need_ws(ws, ws_bytes, forward_ws(cfg)));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const moe_config_t *c = cfg;
    const size_t T = (size_t)c->num_tokens, E = (size_t)c->num_experts, S = T * c->top_k, d = (size_t)c->d_model;
    Carve cv{static_cast<uint8_t *>(ws)};
    void *ws_route = cv.take<uint8_t>(route_ws(c));
    void *ws_perm = cv.take<uint8_t>(permute_ws(c));
    void *ws_ffn = cv.take<uint8_t>(ffn_ws(c));
    void *ws_shared = cv.take<uint8_t>(shared_ws(c));
    void *x_perm = cv.take<uint8_t>(S * d * elem_bytes(c));
    float *y_perm = cv.take<float>(S * d * 4);
    float *z = c->num_shared ? cv.take<float>(T * d * 4) : nullptr;
    moe_forward_io_t o{};
    if (io) o = *io;
    float *logits_ws = cv.take<float>(T * E * 4);
    int32_t *idx_ws = cv.take<int32_t>(S * 4);
    float *w_ws = cv.take<float>(S * 4);
    int32_t *perm_ws = cv.take<int32_t>(S * 4);
    int32_t *inv_ws = cv.take<int32_t>(S * 4);
    float *lse_ws = cv.take<float>(T * 4);
    float *P_ws = cv.take<float>(E * 4);
    int32_t *cnt_ws = cv.take<int32_t>(E * 4);
    int32_t *kept_ws = cv.take<int32_t>(E * 4);
    float *f_ws = cv.take<float>(E * 4);
    int32_t *off_ws = cv.take<int32_t>((E + 1) * 4);
    moe_stats_t *st_ws = cv.take<moe_stats_t>(sizeof(moe_stats_t));
    if (!o.logits) o.logits = logits_ws;
    if (!o.topk_idx) o.topk_idx = idx_ws;
    if (!o.topk_w) o.topk_w = w_ws;
    if (!o.perm) o.perm = perm_ws;
    if (!o.inv) o.inv = inv_ws;
    if (!o.lse) o.lse = lse_ws;
    if (!o.prob_mean) o.prob_mean = P_ws;
    if (!o.counts) o.counts = cnt_ws;
    if (!o.kept) o.kept = kept_ws;
    if (!o.f) o.f = f_ws;
    if (!o.offsets) o.offsets = off_ws;
    if (!o.stats) o.stats = st_ws;
    if (o.x_perm) x_perm = o.x_perm;
    if (o.hidden) ws_ffn = o.hidden;
    if (o.y_perm) y_perm = o.y_perm;
    if (o.shared_hidden) ws_shared = o.shared_hidden;

    void *const *ev = o.stage_events;
    auto mark = [&](int i) {
        if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
    };
    mark(0);
    if (given_idx) {
        // routing given by the caller (hash routing or any other source)
        o.topk_idx = const_cast<int32_t *>(given_idx);
        o.topk_w = const_cast<float *>(given_w);
    } else {
        TRY(route_impl(c, x, w->w_router, w->b_router, c->score_fn == MOE_SCORE_SIGMOID ? sel_bias : nullptr,
                       o.logits, nullptr, o.topk_idx, o.topk_w, o.lse, o.prob_mean, o.counts, ws_route, s,
                       /*reduce=*/false));
    }
    mark(1);
    TRY(permute_impl(c, x, o.topk_idx, o.counts, o.kept, o.offsets, o.perm, o.inv, x_perm, ws_perm, s));
    mark(2);
    // bf16 layer without saved expert outputs (not a training forward, y_perm
    // not requested): the second expert GEMM's epilogue applies the gates and
    // adds the residual to each token's first kept row, so the combine reads
    // no x and multiplies nothing
    const bool prep = c->dtype == MOE_DTYPE_BF16 && !o.pre_act && !(io && io->y_perm);
    CombinePrep cp{};
    if (prep) {
        cp.perm = o.perm;
        cp.gate = o.topk_w;
        cp.inv = o.inv;
        cp.x = c->residual ? static_cast<const bf16 *>(x) : nullptr;
        cp.k = c->top_k;
    }
    TRY(ffn_impl(c, x_perm, (int64_t)S, o.offsets, c->num_experts, 0, w->w1, w->b1, w->w3, w->w2, w->b2, ws_ffn,
                 y_perm, s, ev ? ev[3] : nullptr, o.pre_act, prep ? &cp : nullptr));
    mark(4);
    if (c->num_shared)
        TRY(ffn_impl(c, x, (int64_t)T, nullptr, 1, (int)T, w->shared_w1, nullptr, w->shared_w3, w->shared_w2,
                     nullptr, ws_shared, z, s, nullptr, o.shared_pre_act));
    mark(5);
    if (prep)
        TRY(cuda_status(launch_combine_prepped(c->num_tokens, c->d_model, c->top_k, c->dtype, y_perm, o.inv, z,
                                               c->residual ? x : nullptr, out, s),
                        "combine launch"));
    else
        TRY(cuda_status(launch_combine(c->num_tokens, c->d_model, c->top_k, c->dtype, y_perm, o.inv, o.topk_w, z,
                                       c->residual ? x : nullptr, out, s),
                        "combine launch"));
    mark(6);
    StatsParams sp{};
    sp.T = c->num_tokens;
    sp.E = c->num_experts;
    sp.k = c->top_k;
    sp.cap = capacity_of(c);
    sp.drop = c->drop_tokens;
    sp.counts = o.counts;
    sp.kept = o.kept;
    if (!given_idx) {
        // P and z from the router's per-block partials (prob_mean written here)
        const RoutePartials rp = route_partials(c, ws_route);
        sp.part_prob = rp.prob;
        sp.part_z = rp.z;
        sp.nblk = rp.nblk;
        sp.prob_out = o.prob_mean;
    }
    sp.f = o.f;
    sp.stats = o.stats;
    TRY(cuda_status(launch_stats(sp, s), "stats launch"));
    mark(7);
    return MOE_OK;
}

// K-grouped weight-gradient GEMM: out[g] (M x N, fp32) = A[:, K_g] B[:, K_g]^T
// with A [M, Kp], B [N, Kp] bf16 K-major and K_g = pad[g] .. pad[g+1]-1.
moe_status_t wgrad_gemm(const bf16 *A, int M, const bf16 *B, int N, int64_t Kp, const int32_t *pad, int G,
                        float *out, cudaStream_t s) {
    GemmProblem g{};
    g.A = A;
    g.a_rows = M;
    g.B = B;
    g.b_rows_total = N;
    g.b_group_rows = 0;
    g.seg = pad;
    g.G = G;
    g.M = M;
    g.N = N;
    g.K = (int)Kp;
    g.out = out;
    g.ldo = N;
    g.out_f32 = 1;
    g.kgroup = 1;
    g.out_group_stride = (int64_t)M * N;
    return cuda_status(launch_grouped_gemm(g, s), "weight-gradient GEMM launch");
}

// K-grouped weight-gradient GEMM with both operands read in place (MN-major):
// out[g] (M x N, fp32) = A[rows_g, :M]^T B[rows_g, :N], rows_g = seg[g] ..
// seg[g+1]-1 of the row-major A (row stride lda) and B (ldb); K = rows.
moe_status_t wgrad_gemm_rows(const bf16 *A, int64_t lda, int M, const bf16 *B, int64_t ldb, int N, int64_t rows,
                             const int32_t *seg, int G, float *out, cudaStream_t s) {
    GemmProblem g{};
    g.A = A;
    g.a_rows = rows;
    g.B = B;
    g.b_rows_total = rows;
    g.seg = seg;
    g.G = G;
    g.M = M;
    g.N = N;
    g.K = (int)rows;
    g.out = out;
    g.ldo = N;
    g.out_f32 = 1;
    g.kgroup = 1;
    g.kg_mn = 1;
    g.lda = lda;
    g.ldb = ldb;
    g.out_group_stride = (int64_t)M * N;
    return cuda_status(launch_grouped_gemm(g, s), "weight-gradient GEMM launch");
}

// M-grouped data-gradient GEMM with the weights read in place (MN-major B):
// out rows of group g = A rows x W_g, W stored [G * K_g rows, N cols]; with
// B2 the K columns from k_split on come from B2 (the [W1 | W3] stack).
moe_status_t dgrad_gemm(const bf16 *A, int64_t a_rows, const int32_t *seg, int G, int M, const bf16 *B,
                        const bf16 *B2, int k_split, int b_group_rows, int N, int K, void *out, int out_f32,
                        int64_t ldo, bf16 *pre, int64_t ld_pre, int epi_bwd, int act, cudaStream_t s) {
    GemmProblem g{};
    g.A = A;
    g.a_rows = a_rows;
    g.B = B;
    g.B2 = B2;
    g.k_split = k_split;
    g.b_mn = 1;
    g.b_rows_total = (int64_t)G * b_group_rows;
    g.b_group_rows = b_group_rows;
    g.seg = seg;
    g.G = G;
    g.M = M;
    g.N = N;
    g.K = K;
    g.out = out;
    g.ldo = ldo;
    g.out_f32 = out_f32;
    g.pre = pre;
    g.ld_pre = ld_pre;
    g.epi_bwd = epi_bwd;
    g.act = act;
    return cuda_status(launch_grouped_gemm(g, s), "data-gradient GEMM launch");
}

moe_status_t backward_impl(const moe_config_t *c, const moe_weights_t *w, const void *x, const void *dout,
                           const moe_saved_t *sv, float aux_coef, float z_coef, const moe_grads_t *gr,
                           void *const *ev, void *ws, cudaStream_t s) {
    auto mark = [&](int i) {
        if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
    };
    const BwdDims b = bwd_dims(c);
    const bool gated = c->activation == MOE_ACT_SWIGLU;
    const int act = c->activation == MOE_ACT_GELU ? 1 : (c->activation == MOE_ACT_RELU ? 2 : 0);
    const int epi = gated ? 1 : 2;
    const int E = (int)b.E, d = (int)b.d, F = (int)b.F, nF = (int)b.nF;
    Carve cv{static_cast<uint8_t *>(ws)};
    bf16 *dy = cv.take<bf16>(b.R * b.d * 2);
    float *dgate = cv.take<float>(b.T * b.k * 4);
    float *dl = cv.take<float>(b.T * b.E * 4);
    int32_t *pad = cv.take<int32_t>((b.E + 1) * 4);
    int32_t *pad1 = cv.take<int32_t>(2 * 4);
    bf16 *da = cv.take<bf16>(b.R * b.nF * 2);
    float *dxp = cv.take<float>(b.R * b.d * 4);
    float *rwpart = cv.take<float>((size_t)router_wgrad_chunks(b.T) * b.E * b.d * 4);
    const bool wide = wide_router(c);
    bf16 *dl_hi = wide ? cv.take<bf16>(b.T * b.E * 2) : nullptr;
    bf16 *dl_lo = wide ? cv.take<bf16>(b.T * b.E * 2) : nullptr;
    float *dxr = wide ? cv.take<float>(b.T * b.d * 4) : nullptr;
    bf16 *dlT2 = wide ? cv.take<bf16>(b.E * 2 * b.Tp * 2) : nullptr;
    bf16 *xT2 = wide ? cv.take<bf16>(b.d * 2 * b.Tp * 2) : nullptr;
    int32_t *pad2 = wide ? cv.take<int32_t>(2 * 4) : nullptr;
    const bf16 *W1 = static_cast<const bf16 *>(w->w1), *W3 = static_cast<const bf16 *>(w->w3);
    const bf16 *W2 = static_cast<const bf16 *>(w->w2);
    const bf16 *go = static_cast<const bf16 *>(dout);
#define CU(call, what) TRY(cuda_status((call), what))
    mark(0);
    // combine and router backward
    CU(launch_combine_bwd(b.T, d, (int)b.k, go, sv->topk_w, sv->inv, sv->y_perm, dy, dgate, s), "combine backward");
    CU(launch_router_bwd(b.T, E, (int)b.k, c->score_fn, c->renormalize, sv->logits, sv->topk_idx, dgate, sv->counts,
                         aux_coef, z_coef, dl, dl_hi, dl_lo, s),
       "router backward");
    if (wide) {
        // dx's router term dlogits W_r on the tensor cores (K = E, W_r read in place)
        TRY(dgrad_gemm(dl_hi, b.T, nullptr, 1, (int)b.T, static_cast<const bf16 *>(w->w_router), nullptr, E, E, d,
                       E, dxr, 1, d, nullptr, 0, 0, 0, s));
    }
    mark(1);
    // dh = dy W2 -> da (activation backward in the epilogue); dx_perm = da [W1 | W3]
    TRY(dgrad_gemm(dy, b.R, sv->offsets, E, 0, W2, nullptr, d, d, F, d, da, 0, nF,
                   const_cast<bf16 *>(static_cast<const bf16 *>(sv->pre_act)), nF, epi, act, s));
    mark(2);
    TRY(dgrad_gemm(da, b.R, sv->offsets, E, 0, W1, gated ? W3 : nullptr, F, F, d, nF, dxp, 1, d, nullptr, 0, 0, 0,
                   s));
    mark(3);
    // shared expert: gate 1, A = dout
    float *dxs = nullptr;
    bf16 *das = nullptr;
    if (c->num_shared) {
        das = cv.take<bf16>(b.T * b.nF * 2);
        dxs = cv.take<float>(b.T * b.d * 4);
        const bf16 *SW1 = static_cast<const bf16 *>(w->shared_w1), *SW3 = static_cast<const bf16 *>(w->shared_w3);
        TRY(dgrad_gemm(go, b.T, nullptr, 1, (int)b.T, static_cast<const bf16 *>(w->shared_w2), nullptr, d, d, F, d,
                       das, 0, nF, const_cast<bf16 *>(static_cast<const bf16 *>(sv->shared_pre_act)), nF, epi, act,
                       s));
        TRY(dgrad_gemm(das, b.T, nullptr, 1, (int)b.T, SW1, gated ? SW3 : nullptr, F, F, d, nF, dxs, 1, d, nullptr,
                       0, 0, 0, s));
    }
    mark(4);
    CU(launch_dx_assemble(b.T, d, (int)b.k, E, dxp, sv->inv, go, c->residual, dxs, dl,
                          static_cast<const bf16 *>(w->w_router), dxr, gr->dx, s),
       "dx assembly");
    mark(5);
    // weight gradients over the experts' rows, read in place (K = the rows)
    const bf16 *XP = static_cast<const bf16 *>(sv->x_perm), *H = static_cast<const bf16 *>(sv->hidden);
    if (gr->dw2) TRY(wgrad_gemm_rows(dy, d, d, H, F, F, b.R, sv->offsets, E, gr->dw2, s));
    mark(6);
    if (gr->dw1) TRY(wgrad_gemm_rows(da, nF, F, XP, d, d, b.R, sv->offsets, E, gr->dw1, s));
    if (gated && gr->dw3) TRY(wgrad_gemm_rows(da + F, nF, F, XP, d, d, b.R, sv->offsets, E, gr->dw3, s));
    mark(7);
    if (!gated && gr->db1) CU(launch_group_colsum(da, nF, sv->offsets, E, F, gr->db1, s), "db1");
    if (!gated && gr->db2) CU(launch_group_colsum(dy, d, sv->offsets, E, d, gr->db2, s), "db2");
    const int Ti = (int)b.T;
    if (wide) {
        CU(launch_pad_offsets(nullptr, 1, Ti, pad1, s), "token padded offsets");
        // dW_r = dlogits^T x on the tensor cores, one group over K = 2 Tp:
        // [hi | lo]^T against [x^T | x^T], so dlogits keeps ~16 bits
        CU(launch_pad_offsets(nullptr, 1, 2 * (int)b.Tp, pad2, s), "router K offsets");   // {0, 2 Tp}
        CU(launch_transpose_pack(dl_hi, E, E, nullptr, pad1, 1, Ti, b.Tp, dlT2, 2 * b.Tp, s), "dlogits hi pack");
        CU(launch_transpose_pack(dl_lo, E, E, nullptr, pad1, 1, Ti, b.Tp, dlT2 + b.Tp, 2 * b.Tp, s),
           "dlogits lo pack");
        CU(launch_transpose_pack(static_cast<const bf16 *>(x), d, d, nullptr, pad1, 1, Ti, b.Tp, xT2, 2 * b.Tp, s),
           "x pack");
        CU(launch_transpose_pack(static_cast<const bf16 *>(x), d, d, nullptr, pad1, 1, Ti, b.Tp, xT2 + b.Tp,
                                 2 * b.Tp, s),
           "x pack");
        if (gr->dw_router) TRY(wgrad_gemm(dlT2, E, xT2, d, 2 * b.Tp, pad2, 1, gr->dw_router, s));
        CU(launch_router_wgrad(b.T, d, E, dl, static_cast<const bf16 *>(x), rwpart, nullptr, gr->db_router, s),
           "router bias gradient");
    } else {
        CU(launch_router_wgrad(b.T, d, E, dl, static_cast<const bf16 *>(x), rwpart, gr->dw_router, gr->db_router,
                               s),
           "router weight gradient");
    }
    if (c->num_shared && (gr->shared_dw1 || gr->shared_dw2 || gr->shared_dw3)) {
        // one group: all T tokens
        CU(launch_fill_range(pad, Ti, s), "token range");
        const bf16 *SH = static_cast<const bf16 *>(sv->shared_hidden), *X = static_cast<const bf16 *>(x);
        if (gr->shared_dw2) TRY(wgrad_gemm_rows(go, d, d, SH, F, F, b.T, pad, 1, gr->shared_dw2, s));
        if (gr->shared_dw1) TRY(wgrad_gemm_rows(das, nF, F, X, d, d, b.T, pad, 1, gr->shared_dw1, s));
        if (gated && gr->shared_dw3) TRY(wgrad_gemm_rows(das + F, nF, F, X, d, d, b.T, pad, 1, gr->shared_dw3, s));
    }
#undef CU
    mark(8);
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_forward(const moe_config_t *cfg, const moe_weights_t *weights, const void *x, const float *sel_bias,
                         void *out, const moe_forward_io_t *io, void *ws, size_t ws_bytes, moe_stream_t stream) {
    return forward_impl(cfg, weights, x, sel_bias, nullptr, nullptr, out, io, ws, ws_bytes, stream);
}

moe_status_t moe_forward_from_routing(const moe_config_t *cfg, const moe_weights_t *weights, const void *x,
                                      const int32_t *topk_idx, const float *topk_w, void *out,
                                      const moe_forward_io_t *io, void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t S = cfg->num_tokens * cfg->top_k;
    TRY(need(topk_idx, "topk_idx", S));
    TRY(need(topk_w, "topk_w", S));
    return forward_impl(cfg, weights, x, nullptr, topk_idx, topk_w, out, io, ws, ws_bytes, stream);
}

moe_status_t moe_route_hash(const moe_config_t *cfg, const int32_t *token_ids, int32_t *topk_idx, float *topk_w,
                            moe_stream_t stream) {
    TRY(check_cfg(cfg));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    TRY(need(token_ids, "token_ids", T));
    TRY(need(topk_idx, "topk_idx", S));
    TRY(need(topk_w, "topk_w", S));
    return cuda_status(launch_route_hash(T, cfg->num_experts, cfg->top_k, token_ids, topk_idx, topk_w,
                                         static_cast<cudaStream_t>(stream)),
                       "moe_route_hash launch");
}

moe_status_t moe_backward(const moe_config_t *cfg, const moe_weights_t *weights, const void *x, const void *dout,
                          const moe_saved_t *saved, const moe_grads_t *grads, const moe_backward_opts_t *opts,
                          void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    if (cfg->dtype != MOE_DTYPE_BF16) return fail(MOE_ERR_UNSUPPORTED, "moe_backward needs a bf16 layer");
    moe_backward_opts_t o{};
    if (opts) o = *opts;
    if (!isfinite(o.aux_coef) || !isfinite(o.z_coef)) return fail(MOE_ERR_INVALID_ARG, "coefficients must be finite");
    TRY(need(weights, "weights"));
    TRY(need(saved, "saved"));
    TRY(need(grads, "grads"));
    const int64_t T = cfg->num_tokens, S = T * cfg->top_k;
    const bool gated = cfg->activation == MOE_ACT_SWIGLU;
    TRY(need16(x, "x", T));
    TRY(need16(dout, "dout", T));
    TRY(need16(weights->w_router, "w_router"));
    TRY(check_weights_ffn(cfg, weights->w1, weights->w3, weights->w2));
    if (cfg->num_shared) TRY(check_weights_ffn(cfg, weights->shared_w1, weights->shared_w3, weights->shared_w2));
    TRY(need(saved->topk_idx, "saved topk_idx", S));
    TRY(need(saved->topk_w, "saved topk_w", S));
    TRY(need(saved->logits, "saved logits", T));
    TRY(need(saved->inv, "saved inv", S));
    TRY(need(saved->offsets, "saved offsets"));
    TRY(need(saved->counts, "saved counts"));
    TRY(need16(saved->x_perm, "saved x_perm", S));
    TRY(need16(saved->pre_act, "saved pre_act", S));
    TRY(need16(saved->hidden, "saved hidden", S));
    TRY(need16(saved->y_perm, "saved y_perm", S));
    if (cfg->num_shared) {
        TRY(need16(saved->shared_pre_act, "saved shared_pre_act", T));
        TRY(need16(saved->shared_hidden, "saved shared_hidden", T));
    }
    TRY(need16(grads->dx, "grads dx", T));
    if (!gated && grads->dw3) return fail(MOE_ERR_INVALID_ARG, "grads dw3 given for a layer without W3");
    TRY(need_ws(ws, ws_bytes, bwd_ws(cfg)));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // no tokens: every weight gradient is zero
        const size_t E = cfg->num_experts, d = cfg->d_model, F = cfg->d_ff;
        struct { float *p; size_t n; } z[] = {
            {grads->dw_router, E * d}, {grads->db_router, E}, {grads->dw1, E * F * d}, {grads->db1, E * F},
            {grads->dw3, E * F * d}, {grads->dw2, E * d * F}, {grads->db2, E * d}, {grads->shared_dw1, F * d},
            {grads->shared_dw3, F * d}, {grads->shared_dw2, d * F}};
        for (auto &q : z)
            if (q.p) TRY(cuda_status(cudaMemsetAsync(q.p, 0, q.n * sizeof(float), s), "zero gradients"));
        return MOE_OK;
    }
    return backward_impl(cfg, weights, x, dout, saved, o.aux_coef, o.z_coef, grads, o.stage_events, ws, s);
}

moe_status_t moe_ec_capacity(const moe_config_t *cfg, int64_t *capacity) {
    TRY(check_cfg(cfg));
    TRY(check_ec(cfg));
    TRY(need(capacity, "capacity"));
    *capacity = ec_capacity_of(cfg);
    return MOE_OK;
}

moe_status_t moe_route_expert_choice(const moe_config_t *cfg, const float *logits, int32_t *row_token,
                                     int32_t *tok_row, float *tok_gate, int32_t *offsets, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    TRY(check_ec(cfg));
    const int64_t T = cfg->num_tokens, TE = T * cfg->num_experts;
    TRY(need(logits, "logits", TE));
    TRY(need(row_token, "row_token", ec_capacity_of(cfg) * cfg->num_experts));
    TRY(need(tok_row, "tok_row", TE));
    TRY(need(tok_gate, "tok_gate", TE));
    TRY(need(offsets, "offsets"));
    return ec_route_impl(cfg, logits, row_token, tok_row, tok_gate, offsets, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_forward_expert_choice(const moe_config_t *cfg, const moe_weights_t *w, const void *x, void *out,
                                       const moe_ec_io_t *io, void *ws, size_t ws_bytes, moe_stream_t stream) {
    TRY(check_cfg(cfg));
    TRY(check_ec(cfg));
    TRY(need(w, "weights"));
    TRY(need16(x, "x", cfg->num_tokens));
    TRY(need16(out, "out", cfg->num_tokens));
    TRY(need16(w->w_router, "w_router"));
    TRY(check_weights_ffn(cfg, w->w1, w->w3, w->w2));
    TRY(check_bias(w->b1));
    TRY(check_bias(w->b2));
    if (cfg->num_shared) TRY(check_weights_ffn(cfg, w->shared_w1, w->shared_w3, w->shared_w2));
    TRY(need_ws(ws, ws_bytes, ec_ws(cfg)));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const moe_config_t *c = cfg;
    const size_t T = (size_t)c->num_tokens, E = (size_t)c->num_experts, d = (size_t)c->d_model;
    const int64_t Cap = ec_capacity_of(c);
    const size_t R = E * (size_t)Cap;
    Carve cv{static_cast<uint8_t *>(ws)};
    moe_ec_io_t o{};
    if (io) o = *io;
    float *logits_ws = cv.take<float>(T * E * 4);
    int32_t *tok_row_ws = cv.take<int32_t>(T * E * 4);
    float *gate_ws = cv.take<float>(T * E * 4);
    int32_t *row_token_ws = cv.take<int32_t>(R * 4);
    int32_t *off_ws = cv.take<int32_t>((E + 1) * 4);
    void *x_perm = cv.take<uint8_t>(R * d * elem_bytes(c));
    void *H = cv.take<uint8_t>(R * (size_t)c->d_ff * elem_bytes(c));
    float *y_perm = cv.take<float>(R * d * 4);
    void *ws_shared = c->num_shared ? cv.take<uint8_t>(shared_ws(c)) : nullptr;
    float *z = c->num_shared ? cv.take<float>(T * d * 4) : nullptr;
    if (!o.logits) o.logits = logits_ws;
    if (!o.tok_row) o.tok_row = tok_row_ws;
    if (!o.tok_gate) o.tok_gate = gate_ws;
    if (!o.row_token) o.row_token = row_token_ws;
    if (!o.offsets) o.offsets = off_ws;
    void *const *ev = o.stage_events;
    auto mark = [&](int i) {
        if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
    };
    mark(0);
    TRY(router_logits_impl(c, x, w->w_router, w->b_router, o.logits, s));
    TRY(ec_route_impl(c, o.logits, o.row_token, o.tok_row, o.tok_gate, o.offsets, s));
    mark(1);
    TRY(cuda_status(launch_gather_rows(x, c->num_tokens, o.row_token, (int64_t)R, c->d_model, c->dtype, x_perm, s),
                    "expert-choice gather launch"));
    mark(2);
    TRY(ffn_impl(c, x_perm, (int64_t)R, o.offsets, c->num_experts, 0, w->w1, w->b1, w->w3, w->w2, w->b2, H, y_perm,
                 s, ev ? ev[3] : nullptr));
    mark(4);
    if (c->num_shared)
        TRY(ffn_impl(c, x, (int64_t)T, nullptr, 1, (int)T, w->shared_w1, nullptr, w->shared_w3, w->shared_w2,
                     nullptr, ws_shared, z, s));
    mark(5);
    TRY(cuda_status(launch_combine(c->num_tokens, c->d_model, c->num_experts, c->dtype, y_perm, o.tok_row,
                                   o.tok_gate, z, c->residual ? x : nullptr, out, s),
                    "expert-choice combine launch"));
    mark(6);
    mark(7);
    return MOE_OK;
}

moe_status_t moe_set_option(int32_t option, int64_t value) {
    if (!set_option(option, value))
        return fail(MOE_ERR_INVALID_ARG, "moe_set_option: unknown option %d or value %lld out of range", option,
                    (long long)value);
    return MOE_OK;
}

moe_status_t moe_get_option(int32_t option, int64_t *value) {
    TRY(need(value, "value"));
    if (!get_option(option, value)) return fail(MOE_ERR_INVALID_ARG, "moe_get_option: unknown option %d", option);
    return MOE_OK;
}

moe_status_t moe_check_device_error(int32_t *code) {
    TRY(need(code, "code"));
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_status(e, "cudaDeviceSynchronize");
    int32_t *flag = device_error_flag();
    if (!flag) return fail(MOE_ERR_CUDA, "device error flag unavailable");
    int32_t v = 0;
    e = cudaMemcpy(&v, flag, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e, "read device error flag");
    if (v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpy(flag, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_status(e, "clear device error flag");
    }
    *code = v;
    return MOE_OK;
}

}  // extern "C"
