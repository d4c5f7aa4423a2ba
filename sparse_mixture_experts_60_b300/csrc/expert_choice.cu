// Expert-choice routing: every expert takes the C tokens with the largest
// router logit for it ("MoE Training: Mixture of Experts", Core Concepts,
// Routing Mechanisms, Expert Choice Routing: the router's scores are
// transposed to [experts, tokens] and each expert keeps its top
// capacity-per-expert tokens).
//
// Selection, one CTA per expert: the expert's logit column is turned into
// order-preserving 32-bit keys (held in shared memory when the batch fits),
// the C-th largest key tau is found by an MSB-first radix select (four
// passes of 8-bit digits over a 256-bin shared histogram, warp-aggregated
// with match_any), and one pass in token order with block-wide exclusive
// scans takes every token above tau plus the lowest-index tokens equal to
// it.  The expert's rows e*C .. e*C+C-1 hold its tokens in token order.
// The selection is unique, so it is bit-exact against any implementation
// fed the same fp32 logits.
//
// Gates, warp per token: the softmax probability of the expert over the
// token's logits, for the pairs that were chosen.
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreadsEC = 1024;
constexpr int64_t kEcSmemKeys = 40960;   // keys cached in shared memory (160 KB)

// larger float -> larger unsigned key (finite inputs; -0 and +0 are equal)
__device__ __forceinline__ uint32_t ordered_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// exclusive scan of one int per thread over the CTA; *total = CTA sum
__device__ __forceinline__ int block_exclusive_scan(int v, int *total, int *warp_buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += u;
    }
    __syncthreads();
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? warp_buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += u;
        }
        warp_buf[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    *total = warp_buf[nw - 1];
    return (warp > 0 ? warp_buf[warp - 1] : 0) + x - v;
}

__global__ void __launch_bounds__(kThreadsEC) ec_select_kernel(const float *__restrict__ logits, int64_t T, int E,
                                                              int64_t C, int cache, int32_t *row_token,
                                                              int32_t *tok_row, int32_t *offsets) {
    PDL_ENTER();
    extern __shared__ uint32_t skey[];
    __shared__ unsigned int hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remaining;
    __shared__ int warp_buf[32];
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31;
    if (cache)
        for (int64_t t = threadIdx.x; t < T; t += blockDim.x) skey[t] = ordered_key(__ldg(logits + t * E + e));
    auto key = [&](int64_t t) -> uint32_t { return cache ? skey[t] : ordered_key(__ldg(logits + t * E + e)); };

    uint32_t prefix = 0, mask = 0;
    int remaining = (int)C;   // 1 <= C <= T
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        // whole-CTA steps, so every warp is complete for match_any
        for (int64_t base = 0; base < T; base += blockDim.x) {
            const int64_t t = base + threadIdx.x;
            const uint32_t u = t < T ? key(t) : 0u;
            const bool hit = t < T && (u & mask) == prefix;
            const unsigned bin = hit ? ((u >> shift) & 255u) : 256u;
            const unsigned peers = __match_any_sync(kFull, bin);
            if (hit && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int cum = 0;
            for (int b = 255; b >= 0; --b) {
                if (cum + (int)hist[b] >= remaining) {
                    s_prefix = prefix | ((uint32_t)b << shift);
                    s_remaining = remaining - cum;
                    break;
                }
                cum += (int)hist[b];
            }
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        mask |= 0xffu << shift;
    }
    // tau = key of the C-th largest; `remaining` of the tokens equal to it are taken
    const uint32_t tau = prefix;
    int carry_eq = 0, carry_sel = 0;
    for (int64_t base = 0; base < T; base += blockDim.x) {
        const int64_t t = base + threadIdx.x;
        const bool valid = t < T;
        const uint32_t u = valid ? key(t) : 0u;
        const int is_eq = (valid && u == tau) ? 1 : 0;
        int tot_eq, tot_sel;
        const int eq_rank = carry_eq + block_exclusive_scan(is_eq, &tot_eq, warp_buf);
        const int sel = (valid && (u > tau || (is_eq && eq_rank < remaining))) ? 1 : 0;
        const int pos = carry_sel + block_exclusive_scan(sel, &tot_sel, warp_buf);
        if (valid) {
            const bool take = sel && pos < C;   // pos < C always holds; the test keeps writes in bounds
            const int32_t row = (int32_t)((int64_t)e * C + pos);
            if (take) row_token[row] = (int32_t)t;
            tok_row[t * E + e] = take ? row : -1;
        }
        carry_eq += tot_eq;
        carry_sel += tot_sel;
    }
    if (threadIdx.x == 0) {
        offsets[e] = (int32_t)((int64_t)e * C);
        if (e == E - 1) offsets[E] = (int32_t)((int64_t)E * C);
    }
}

// warp per token: gate = softmax(logits[t])[e] for the chosen pairs
__global__ void __launch_bounds__(256) ec_gate_kernel(const float *__restrict__ logits,
                                                      const int32_t *__restrict__ tok_row, int64_t T, int E,
                                                      float *__restrict__ tok_gate) {
    PDL_ENTER();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *lr = logits + t * E;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, __ldg(lr + e));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    float s = 0.0f;
    for (int e = lane; e < E; e += 32) s += expf(__ldg(lr + e) - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    for (int e = lane; e < E; e += 32)
        tok_gate[t * E + e] = __ldg(tok_row + t * E + e) >= 0 ? expf(__ldg(lr + e) - m) / s : 0.0f;
}

// warp per row: x_perm[r] = x[row_token[r]] (16-byte vectors, four in flight)
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ x,
                                                          const int32_t *__restrict__ row_token, int64_t rows,
                                                          int64_t T, int nvec, uint4 *__restrict__ x_perm,
                                                          int32_t *err) {
    PDL_ENTER();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int32_t tok = __ldg(row_token + r);
    if (tok < 0 || tok >= T) {   // not a token of this batch: row left as is, error flagged
        if (lane == 0) atomicCAS(err, 0, 1);
        return;
    }
    const uint4 *src = x + (int64_t)tok * nvec;
    uint4 *dst = x_perm + r * nvec;
    int v = lane;
    for (; v + 96 < nvec; v += 128) {
        uint4 q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __ldg(src + v + 32 * i);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[v + 32 * i] = q[i];
    }
    for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
}

__global__ void add_bias_kernel(float *logits, const float *b, int64_t T, int E) {
    PDL_ENTER();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < T * E) logits[i] += b[i % E];
}

}  // namespace

cudaError_t launch_ec_select(const float *logits, int64_t T, int E, int64_t C, int32_t *row_token, int32_t *tok_row,
                             int32_t *offsets, cudaStream_t s) {
    if (T == 0) return cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * sizeof(int32_t), s);
    const int cache = T <= kEcSmemKeys ? 1 : 0;
    const size_t smem = cache ? (size_t)T * sizeof(uint32_t) : 0;
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(kEcSmemKeys * sizeof(uint32_t)));
        if (err != cudaSuccess) return err;
    }
    return launch_pdl(ec_select_kernel, dim3((unsigned)E), dim3(kThreadsEC), smem, s, logits, T, E, C, cache,
                      row_token, tok_row, offsets);
}

cudaError_t launch_ec_gates(const float *logits, const int32_t *tok_row, int64_t T, int E, float *tok_gate,
                            cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(ec_gate_kernel, dim3((unsigned)ceil_div(T, 8)), dim3(256), 0, s, logits, tok_row, T, E, tok_gate);
}

cudaError_t launch_gather_rows(const void *x, int64_t T, const int32_t *row_token, int64_t rows, int d, int dtype,
                               void *x_perm, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int nvec = d * (dtype == 0 ? 4 : 2) / 16;
    return launch_pdl(gather_rows_kernel, dim3((unsigned)ceil_div(rows, 8)), dim3(256), 0, s,
                      static_cast<const uint4 *>(x), row_token, rows, T, nvec, static_cast<uint4 *>(x_perm),
                      device_error_flag());
}

cudaError_t launch_add_bias(float *logits, const float *b, int64_t T, int E, cudaStream_t s) {
    if (T == 0 || !b) return cudaSuccess;
    return launch_pdl(add_bias_kernel, dim3((unsigned)ceil_div(T * E, 256)), dim3(256), 0, s, logits, b, T, E);
}

}  // namespace moe
