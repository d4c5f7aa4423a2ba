// Internal launch interface between the C ABI (moe_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

namespace moe {

using bf16 = __nv_bfloat16;

constexpr int kRouteTokPerCta = 32;   // tokens per router CTA (fixed: partials are deterministic)
constexpr int kPermChunk = 2048;      // priority-ordered slots per permute chunk
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device address of one of the library's __device__ variables on the
// current device, looked up once per (device, context) with that device
// current: a cudaDeviceReset, or a primary context released and created
// again, loads the module again at another address, so the cached address
// is used only while the context it was looked up in is the current one.
struct SymbolCache {
    static constexpr int kDevices = 64;
    std::mutex mu;
    void *ctx[kDevices] = {};
    void *ptr[kDevices] = {};
};
void *symbol_address(SymbolCache &cache, const void *symbol);

// Device error flag shared by every kernel of the library (defined in
// gemm_sm103.cu).  Returns its device address on the current device.
int32_t *device_error_flag();

int num_sms();

// Programmatic dependent launch.  Every kernel of the library is launched
// with launch_pdl and starts with PDL_ENTER() (pdl_wait before its first
// global-memory access, then pdl_trigger): the next kernel on the stream is
// launched as soon as every CTA of this one has started, so its launch and
// prologue overlap this kernel's tail, and griddepcontrol.wait still holds it
// until this grid has completed and its writes are visible.  Without the
// launch attribute (MOE_OPT_PDL set to 0, or launches from other code) both
// instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#define PDL_ENTER()       \
    do {                  \
        ::moe::pdl_wait();    \
        ::moe::pdl_trigger(); \
    } while (0)

bool pdl_enabled();
// Process-wide options of moe_set_option (defined in gemm_sm103.cu).
bool set_option(int option, int64_t value);
bool get_option(int option, int64_t *value);

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
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
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- router
struct RouteParams {
    int64_t T;
    int E, k, d;
    int score_fn;          // 0 softmax, 1 sigmoid
    int renormalize;
    const void *x;         // [T,d] (fused path)
    const void *w_router;  // [E,d]
    const float *b_router; // [E] or null
    const float *sel_bias; // [E] or null
    float *logits;         // [T,E]: output (fused path), input (logits path)
    int logits_add_bias;   // logits path: add b_router and write back
    int32_t *topk_idx;
    float *topk_w;
    float *lse;
    float *part_prob;      // [E, nblk] per-CTA sums of softmax probabilities
    int32_t *part_cnt;     // [E, nblk] per-CTA expert counts
    float *part_z;         // [nblk] per-CTA sums of lse^2, or null
};
// fp32 layers, E <= 32: one kernel computes logits from x on the CUDA cores and routes
cudaError_t launch_router_fused(const RouteParams &p, cudaStream_t s);
// logits given in p.logits (optionally + bias, written back): route only
cudaError_t launch_route_logits(const RouteParams &p, cudaStream_t s);
// logits = x w_r^T on CUDA cores (fp32, or shapes the tensor-core path does not take)
cudaError_t launch_router_logits_simt(const RouteParams &p, int dtype, cudaStream_t s);
// hash routing: fixed token -> expert map from token ids, gate 1/k
cudaError_t launch_route_hash(int64_t T, int E, int k, const int32_t *token_ids, int32_t *topk_idx,
                              float *topk_w, cudaStream_t s);
// deterministic reduction of the per-CTA partials: prob_mean[E], counts[E]
cudaError_t launch_route_reduce(const float *part_prob, const int32_t *part_cnt, int64_t nblk,
                                int E, int64_t T, float *prob_mean, int32_t *counts,
                                cudaStream_t s);

// ----------------------------------------------------------------- permute
struct PermuteParams {
    int64_t T;
    int E, k, d, dtype;
    int64_t cap;           // capacity (T*k when no dropping)
    const void *x;
    const int32_t *topk_idx;
    int32_t *counts, *kept, *offsets, *perm, *inv;
    void *x_perm;
    int32_t *hist;         // [nchunk, E] scratch
    int32_t *base;         // [nchunk, E] scratch
    int32_t *lrank;        // [T*k] scratch: rank of each slot within its chunk (two-launch dispatch)
    int chunked;           // 1: always the chunked kernels (which use hist/base)
};
// Layers up to this many slots and experts dispatch in one CTA without
// scratch; larger ones are faster on the chunked kernels, which spread the
// integer work over many SMs (8192 slots, 128 experts: 16.8 us in the
// two-launch form against 19.3 us with the one-CTA ranking).
constexpr int64_t kSmallSlots = 2048;
constexpr int kSmallExperts = 256;
// Layers whose chunk table (chunks of 512, 1024 or 2048 slots x experts)
// has at most this many entries dispatch in two launches: per-chunk histograms and ranks,
// then the row copy, each of whose CTAs rebuilds the chunk bases and
// offsets from the table in shared memory; larger tables use the separate
// histogram, scan and rank kernels.
constexpr int64_t kTwoPassTable = 8192;
cudaError_t launch_permute(const PermuteParams &p, cudaStream_t s);
// Device address of the file-scope scratch of the allocation-free dispatch
// (looked up once per device, on first use, with that device current).
constexpr int64_t kPermStaticScratchInts = 131072;
int32_t *permute_static_scratch();

// ----------------------------------------------------------------- expert choice
// Each expert takes the C tokens with the largest logit (ties: lower token
// index); rows e*C .. e*C+C-1 hold its tokens in token order.
//   row_token [E*C], tok_row [T,E] (row or -1), offsets [E+1] = e*C.
cudaError_t launch_ec_select(const float *logits, int64_t T, int E, int64_t C, int32_t *row_token, int32_t *tok_row,
                             int32_t *offsets, cudaStream_t s);
// tok_gate [T,E] = softmax(logits[t])[e] where tok_row >= 0, else 0
cudaError_t launch_ec_gates(const float *logits, const int32_t *tok_row, int64_t T, int E, float *tok_gate,
                            cudaStream_t s);
// x_perm[r] = x[row_token[r]] for r < rows (a token outside [0, T) raises the error flag)
cudaError_t launch_gather_rows(const void *x, int64_t T, const int32_t *row_token, int64_t rows, int d, int dtype,
                               void *x_perm, cudaStream_t s);
cudaError_t launch_add_bias(float *logits, const float *b, int64_t T, int E, cudaStream_t s);

// ----------------------------------------------------------------- experts
// Grouped GEMM with fused epilogue on the tensor cores (bf16 in, fp32 acc).
// M-grouped (expert FFNs: rows of A in groups, B per group) or K-grouped
// (weight gradients: the groups split K).
//   out[r, n] = epi( sum_k A[r, k] * B[g*b_rows + n, k] )   for rows r of group g
// gated: B2 is the second weight; epi = silu(acc1) * acc2.
// act: 0 none, 1 GELU, 2 ReLU.  out is bf16 (out_f32 = 0) or fp32.
// Routing epilogue of the router GEMM (E <= 32, one thread per token):
// bias, logits written, top-k, gates, lse and the per-32-token partials.
struct RouteEpilogue {
    const float *b_router;
    const float *sel_bias;
    int k, score_fn, renormalize;
    int32_t *topk_idx;
    float *topk_w, *lse;
    float *part_prob;      // [E, nblk]
    int32_t *part_cnt;     // [E, nblk]
    float *part_z;         // [nblk]
    int64_t nblk;          // ceil(T / kRouteTokPerCta)
};

// Combine preparation in the epilogue of the second expert GEMM (fp32
// output, layer forward): row r of slot s = perm[r] (token t = s / k, rank
// j = s % k) stores gate[s] * y + x[t] when no slot of t before j was kept
// (x: the residual, [T, N] bf16), else gate[s] * y.  perm null: off.
struct CombinePrep {
    const int32_t *perm;
    const float *gate;
    const int32_t *inv;
    const bf16 *x;          // null without residual
    int k;
};

struct GemmProblem {
    const bf16 *A; int64_t a_rows;           // A [a_rows, K]
    const bf16 *B; const bf16 *B2; int64_t b_rows_total; int b_group_rows;
    const int32_t *seg;                      // [G+1] row offsets (device) or null
    int G; int M;                            // M: rows when seg is null
    int N, K;
    void *out; int64_t ldo; int out_f32;
    const bf16 *bias; int64_t bias_stride;   // per group, or null
    int act; int gated;
    const RouteEpilogue *route;              // router GEMM with the routing epilogue, or null
    // training forward: pre-activations stored (gated: [rows, 2N] a1 | a3,
    // else [rows, N] a); activation backward (epi_bwd 1 SwiGLU, 2 GELU /
    // ReLU by act): pre-activations read, out = da ([rows, 2N] for SwiGLU)
    bf16 *pre; int64_t ld_pre; int epi_bwd;
    // K-grouped (weight gradients): A [M, K], B [N, K]; group g sums over
    // K columns seg[g] .. seg[g+1]-1 (multiples of 64) into out + g * out_group_stride
    int kgroup; int64_t out_group_stride;
    // MN-major B (data gradients from the stored weights): B [G * K_g rows,
    // N cols]; group g's K rows start at g * b_group_rows; with B2 the K
    // columns from k_split on come from B2 (the [W1 | W3] stack)
    int b_mn; int k_split;
    // K-grouped with both operands read in place (kg_mn): A [K rows, M
    // cols] (row stride lda), B [K rows, N cols] (ldb); seg[g] .. seg[g+1]-1
    // are group g's rows (any offsets), K the total rows
    int kg_mn; int64_t lda, ldb;
    CombinePrep comb;                        // second expert GEMM of the forward, or zeros
};
cudaError_t launch_grouped_gemm(const GemmProblem &p, cudaStream_t s);
bool grouped_gemm_supported(int N, int K, int gated, int out_f32, int has_bias);

// CUDA-core grouped FFN layer for fp32 storage (same contract as above, fp32).
struct SimtProblem {
    const float *A; const float *B; const float *B2;
    const int32_t *seg; int G; int M; int64_t max_rows;
    int N, K; float *out; int64_t ldo;
    const float *bias; int64_t bias_stride; int act; int gated;
};
cudaError_t launch_ffn_simt(const SimtProblem &p, cudaStream_t s);

// ----------------------------------------------------------------- combine / stats
cudaError_t launch_combine(int64_t T, int d, int k, int dtype, const float *y_perm,
                           const int32_t *inv, const float *topk_w, const float *shared_out,
                           const void *x_res, void *out, cudaStream_t s);
// The combine after a second expert GEMM with CombinePrep: y_perm rows hold
// gate * y (+ x for a token's first kept slot); out = sum of the token's
// kept rows (j ascending) + shared_out, + x only when no slot was kept.
cudaError_t launch_combine_prepped(int64_t T, int d, int k, int dtype, const float *y_perm, const int32_t *inv,
                                   const float *shared_out, const void *x_res, void *out, cudaStream_t s);
struct StatsParams {
    int64_t T; int E, k; int64_t cap; int drop;
    const int32_t *counts, *kept; const float *prob_mean, *lse;
    // router partials instead of prob_mean / lse (the layer forward):
    // P_e = sum_blk part_prob[e, blk] / T (written to prob_out when not
    // null), z = sum_blk part_z[blk] / T
    const float *part_prob, *part_z; int64_t nblk; float *prob_out;
    float *f; void *stats;
};
cudaError_t launch_stats(const StatsParams &p, cudaStream_t s);
cudaError_t launch_bias_update(int64_t T, int E, int k, const int32_t *counts, float *bias,
                               float gamma, cudaStream_t s);

// ----------------------------------------------------------------- backward
cudaError_t launch_combine_bwd(int64_t T, int d, int k, const bf16 *dout, const float *topk_w, const int32_t *inv,
                               const float *y, bf16 *dy, float *dgate, cudaStream_t s);
cudaError_t launch_router_bwd(int64_t T, int E, int k, int score_fn, int renormalize, const float *logits,
                              const int32_t *topk_idx, const float *dgate, const int32_t *counts, float aux_coef,
                              float z_coef, float *dl, bf16 *dl_hi, bf16 *dl_lo, cudaStream_t s);
cudaError_t launch_dx_assemble(int64_t T, int d, int k, int E, const float *dx_perm, const int32_t *inv,
                               const bf16 *dout, int residual, const float *dxs, const float *dl,
                               const bf16 *w_router, const float *dxr, float *dx, cudaStream_t s);
int64_t router_wgrad_chunks(int64_t T);   // partial buffer: chunks * E * d floats
cudaError_t launch_router_wgrad(int64_t T, int d, int E, const float *dl, const bf16 *x, float *part, float *dw,
                                float *db, cudaStream_t s);
// out[c * ld_out + pad[g] + i] = in[off[g] + i][c] (zero padding), pad[G] <= max_padded
cudaError_t launch_transpose_pack(const bf16 *in, int ld_in, int cols, const int32_t *off, const int32_t *pad, int G,
                                  int rows, int64_t max_padded, bf16 *out, int64_t ld_out, cudaStream_t s);
cudaError_t launch_pad_offsets(const int32_t *off, int G, int rows, int32_t *pad, cudaStream_t s);
// out[g][c] = sum of in[r][c] over the rows off[g] .. off[g+1]-1 (fp32)
cudaError_t launch_group_colsum(const bf16 *in, int64_t ld, const int32_t *off, int G, int C, float *out,
                                cudaStream_t s);
cudaError_t launch_fill_range(int32_t *seg, int n, cudaStream_t s);   // seg = {0, n}

}  // namespace moe
