// Router: logits, fp32 softmax / sigmoid scores, warp-level top-k in
// registers, gates, logsumexp, and deterministic balance partials.
//
// Pages: "MoE Training: Mixture of Experts" (Quick Start MoELayer: gate
// Linear, softmax, topk, renormalise); "Mixture of Experts (MoE) From
// Scratch to DeepSeek V3" (routing formula h(x) = x W_g, fp32 router,
// sigmoid routing, selection bias b_i); "moe_code.py" (Router,
// MixtureOfExperts steps 1-3).
//
// Layout of the work: a CTA owns 32 consecutive tokens (8 warps x 4).  A
// token's experts are spread over a "group" of G lanes (G = 8, 16 or 32),
// lane r of the group holding experts r, r+G, r+2G, ... (VPL values).  With
// G < 32 one warp routes 32/G tokens at once.  All reductions are xor
// butterflies, so every lane of a group ends with bit-identical values and
// the result does not depend on scheduling.
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"
#include "route_device.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Route one token held by a group of G lanes (VPL logits per lane).
template <int G, int VPL>
__device__ __forceinline__ void route_group(const RouteParams &p, const float (&l)[VPL], int r,
                                            bool tok_ok, int64_t t, float (&psum)[VPL], float &zsum,
                                            int *s_cnt) {
    const int E = p.E, k = p.k;
    float key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = r + G * i;
        float kv = -INFINITY;
        if (e < E) {
            kv = (p.score_fn == 0) ? l[i]
                                   : __fadd_rn(sigmoid_key(l[i]), p.sel_bias ? p.sel_bias[e] : 0.0f);
            if (kv != kv) kv = -INFINITY;
        }
        key[i] = kv;
    }
    // logsumexp of the logits (fp32)
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (r + G * i < E) m = fmaxf(m, l[i]);
    m = group_max<G>(m);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (r + G * i < E) s += expf(l[i] - m);
    s = group_sum<G>(s);
    const float lse = m + logf(s);
    if (tok_ok) {
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (r + G * i < E) psum[i] += expf(l[i] - lse);
        if (r == 0) zsum += lse * lse;
    }
    // top-k: k rounds of a group arg-max over the keys not yet taken
    unsigned taken = 0u;
    int my_e = 0;
    float my_l = 0.0f;
    for (int j = 0; j < k; ++j) {
        float bk = -INFINITY, bl = 0.0f;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = r + G * i;
            if (e < E && !((taken >> i) & 1u) && ranks_before(key[i], e, bk, be)) {
                bk = key[i];
                be = e;
                bl = l[i];
            }
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(kFull, bk, o);
            const int oe = __shfl_xor_sync(kFull, be, o);
            const float ol = __shfl_xor_sync(kFull, bl, o);
            if (ranks_before(ok, oe, bk, be)) {
                bk = ok;
                be = oe;
                bl = ol;
            }
        }
        if (be < E && (be & (G - 1)) == r) taken |= 1u << (be / G);
        if (r == j) {
            my_e = be;
            my_l = bl;
        }
    }
    // gates
    float g = 0.0f;
    if (r < k) g = (p.score_fn == 0) ? expf(my_l - m) : 1.0f / (1.0f + expf(-my_l));
    const float tot = group_sum<G>(g);
    float w;
    if (p.renormalize) w = g / tot;
    else w = (p.score_fn == 0) ? expf(my_l - lse) : g;
    if (tok_ok) {
        if (r < k) {
            p.topk_idx[t * k + r] = my_e;
            p.topk_w[t * k + r] = w;
            atomicAdd(&s_cnt[my_e], 1);
        }
        if (r == 0) p.lse[t] = lse;
    }
}

// Per-CTA partials: psum is summed over the groups of a warp (xor
// butterfly), then over the NW warps in warp order.
template <int G, int VPL, int NW = 8>
__device__ __forceinline__ void write_partials(const RouteParams &p, float (&psum)[VPL], float zsum, int r,
                                               int grp, float *s_prob, const int *s_cnt) {
    __shared__ float s_z[NW];
    const int warp = threadIdx.x >> 5;
    const int EP = G * VPL;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zsum += __shfl_xor_sync(kFull, zsum, o);
    if ((threadIdx.x & 31) == 0) s_z[warp] = zsum;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
#pragma unroll
        for (int o = G; o < 32; o <<= 1) psum[i] += __shfl_xor_sync(kFull, psum[i], o);
        if (grp == 0) s_prob[warp * EP + r + G * i] = psum[i];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        float acc = 0.0f;
        for (int w = 0; w < NW; ++w) acc += s_prob[w * EP + e];
        p.part_prob[(int64_t)e * gridDim.x + blockIdx.x] = acc;   // [E][blocks]
        p.part_cnt[(int64_t)e * gridDim.x + blockIdx.x] = s_cnt[e];
    }
    if (threadIdx.x == 0 && p.part_z) {
        float z = 0.0f;
        for (int w = 0; w < NW; ++w) z += s_z[w];
        p.part_z[blockIdx.x] = z;
    }
}

// 16-byte global load that is not allocated in L1 (read-once stream).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <typename Tin>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
};

// E <= EP <= 32: logits from x on the CUDA cores (the router is read from
// L1, x streamed once with 16-byte loads), then routing in registers.
template <typename Tin, int EP>
__global__ void __launch_bounds__(256, EP <= 16 ? 2 : 1) router_fused_kernel(RouteParams p) {
    PDL_ENTER();
    constexpr int TPW = 32 / EP;            // tokens per warp per round
    constexpr int VN = Vec<Tin>::N;
    __shared__ float s_prob[8 * EP];
    __shared__ int s_cnt[EP];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane % EP, grp = lane / EP;
    const int E = p.E, d = p.d;
    const Tin *x = static_cast<const Tin *>(p.x);
    const Tin *W = static_cast<const Tin *>(p.w_router);
    if (threadIdx.x < EP) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    float psum[1] = {0.0f};
    float zsum = 0.0f;
    const int nvec = d / VN;
    const int64_t cta_t0 = (int64_t)blockIdx.x * kRouteTokPerCta;
#pragma unroll 1
    for (int round = 0; round < 4 / TPW; ++round) {
        const int64_t t0 = cta_t0 + warp * 4 + round * TPW;
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
        // U iterations of x loads are issued before any arithmetic, so each
        // lane keeps U*TPW 16-byte loads in flight (x is streamed past L1,
        // which keeps the router weights resident there)
        constexpr int U = 4;
        for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
            uint4 xr[U][TPW];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int ti = 0; ti < TPW; ++ti) {
                    const int v = v0 + 32 * u;
                    xr[u][ti] = (v < nvec && t0 + ti < p.T)
                                    ? ld_stream(reinterpret_cast<const uint4 *>(x + (t0 + ti) * d) + v)
                                    : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + 32 * u;
                if (v >= nvec) break;
                float xf[TPW][VN];
#pragma unroll
                for (int ti = 0; ti < TPW; ++ti) Vec<Tin>::unpack(xr[u][ti], xf[ti]);
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    if (e < E) {
                        float wf[VN];
                        Vec<Tin>::unpack(__ldg(reinterpret_cast<const uint4 *>(W + (int64_t)e * d) + v), wf);
#pragma unroll
                        for (int ti = 0; ti < TPW; ++ti)
#pragma unroll
                            for (int q = 0; q < VN; ++q)
                                acc[ti * EP + e] = fmaf(xf[ti][q], wf[q], acc[ti * EP + e]);
                    }
                }
            }
        }
        float logit = transpose_reduce32(acc, lane);   // token grp, expert r
        const int64_t t = t0 + grp;
        const bool tok_ok = t < p.T;
        if (r < E) {
            if (p.b_router) logit += p.b_router[r];
            if (tok_ok) p.logits[t * E + r] = logit;
        }
        const float l1[1] = {logit};
        route_group<EP, 1>(p, l1, r, tok_ok, t, psum, zsum, s_cnt);
    }
    __syncthreads();
    write_partials<EP, 1>(p, psum, zsum, r, grp, s_prob, s_cnt);
}

// Routing from logits in memory (optionally adding the router bias and
// writing the biased logits back).  NW warps share a CTA's 32 tokens: a
// token's routing is a chain of dependent shuffles (k arg-max rounds), so
// the wide routers take a warp per token (up to 32 warps) to keep more
// tokens in flight per SM.
template <int G, int VPL, int NW>
__global__ void __launch_bounds__(NW * 32) route_logits_kernel(RouteParams p) {
    PDL_ENTER();
    constexpr int TPR = 32 / G;                       // tokens per warp per round
    constexpr int TPW = kRouteTokPerCta / NW;         // tokens per warp
    static_assert(TPW % TPR == 0 && TPW >= TPR, "tokens per warp");
    extern __shared__ float dyn[];
    float *s_prob = dyn;                                   // [NW][G*VPL]
    int *s_cnt = reinterpret_cast<int *>(dyn + NW * G * VPL);  // [G*VPL]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane % G, grp = lane / G;
    const int E = p.E;
    for (int e = threadIdx.x; e < G * VPL; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    float psum[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) psum[i] = 0.0f;
    float zsum = 0.0f;
    const int64_t cta_t0 = (int64_t)blockIdx.x * kRouteTokPerCta;
#pragma unroll 1
    for (int round = 0; round < TPW / TPR; ++round) {
        const int64_t t = cta_t0 + warp * TPW + round * TPR + grp;
        const bool tok_ok = t < p.T;
        float l[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = r + G * i;
            float v = 0.0f;
            if (tok_ok && e < E) {
                v = p.logits[t * E + e];
                if (p.logits_add_bias && p.b_router) {
                    v += p.b_router[e];
                    p.logits[t * E + e] = v;
                }
            }
            l[i] = v;
        }
        route_group<G, VPL>(p, l, r, tok_ok, t, psum, zsum, s_cnt);
    }
    __syncthreads();
    write_partials<G, VPL, NW>(p, psum, zsum, r, grp, s_prob, s_cnt);
}

// logits = x W^T on CUDA cores, 32x32 output tiles (no bias).
template <typename Tin>
__global__ void __launch_bounds__(256) router_logits_simt_kernel(const Tin *x, const Tin *W,
                                                                 float *logits, int64_t T, int E,
                                                                 int d) {
    PDL_ENTER();
    __shared__ float xs[32][33], ws[32][33];
    const int64_t t0 = (int64_t)blockIdx.x * 32;
    const int e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < d; k0 += 32) {
        for (int i = ty; i < 32; i += 8) {
            const int kk = k0 + tx;
            xs[i][tx] = (t0 + i < T && kk < d) ? (float)x[(t0 + i) * d + kk] : 0.0f;
            ws[i][tx] = (e0 + i < E && kk < d) ? (float)W[(int64_t)(e0 + i) * d + kk] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            const float wv = ws[tx][kk];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(xs[ty + 8 * q][kk], wv, acc[q]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int64_t t = t0 + ty + 8 * q;
        if (t < T && e0 + tx < E) logits[t * E + e0 + tx] = acc[q];
    }
}

// One CTA per expert: fixed strided fp32 sums per thread, then a fixed
// shared-memory tree (deterministic).
__global__ void __launch_bounds__(256) route_reduce_kernel(const float *part_prob, const int32_t *part_cnt,
                                                           int64_t nblk, int E, int64_t T, float *prob_mean,
                                                           int32_t *counts) {
    PDL_ENTER();
    __shared__ float sp[256];
    __shared__ int sc[256];
    const int e = blockIdx.x;
    float s = 0.0f;
    int c = 0;
    for (int64_t b = threadIdx.x; b < nblk; b += blockDim.x) {
        s += part_prob[(int64_t)e * nblk + b];
        c += part_cnt[(int64_t)e * nblk + b];
    }
    sp[threadIdx.x] = s;
    sc[threadIdx.x] = c;
    __syncthreads();
    for (int st = 128; st > 0; st >>= 1) {
        if (threadIdx.x < st) {
            sp[threadIdx.x] += sp[threadIdx.x + st];
            sc[threadIdx.x] += sc[threadIdx.x + st];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        prob_mean[e] = T > 0 ? sp[0] / (float)T : 0.0f;
        counts[e] = sc[0];
    }
}

// Warps per CTA: one token per warp while the registers allow (VPL <= 8:
// 62 registers at 1024 threads), else 16 or 8 warps.
template <int G, int VPL, int NW = (G == 32 ? (VPL <= 8 ? 32 : (VPL <= 16 ? 16 : 8)) : 8)>
cudaError_t launch_route_logits_t(const RouteParams &p, cudaStream_t s) {
    const int64_t nblk = ceil_div(p.T, kRouteTokPerCta);
    const size_t smem = (size_t)(NW * G * VPL) * sizeof(float) + (size_t)(G * VPL) * sizeof(int);
    auto kern = route_logits_kernel<G, VPL, NW>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3((unsigned)nblk), dim3(NW * 32), smem, s, p);
}

// Hash routing: one thread per token.  Choice j of a token is
// fmix32(token_id + j * 0x9E3779B9) mod E (MurmurHash3's 32-bit finalizer,
// a published mixing function), moved to the next free expert, cyclically,
// when an earlier choice of the same token already took it; gate 1/k.
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

__global__ void __launch_bounds__(256) route_hash_kernel(int64_t T, int E, int k, const int32_t *token_ids,
                                                         int32_t *topk_idx, float *topk_w) {
    PDL_ENTER();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const uint32_t id = (uint32_t)token_ids[t];
    int chosen[kMaxTopK];
    const float g = 1.0f / (float)k;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if (j >= k) break;
        int e = (int)(fmix32(id + (uint32_t)j * 0x9E3779B9u) % (uint32_t)E);
        for (;;) {
            bool taken = false;
#pragma unroll
            for (int i = 0; i < kMaxTopK; ++i)
                if (i < j && chosen[i] == e) taken = true;
            if (!taken) break;
            e = (e + 1) % E;
        }
        chosen[j] = e;
        topk_idx[t * k + j] = e;
        topk_w[t * k + j] = g;
    }
}

}  // namespace

cudaError_t launch_route_hash(int64_t T, int E, int k, const int32_t *token_ids, int32_t *topk_idx, float *topk_w,
                              cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(route_hash_kernel, dim3((unsigned)ceil_div(T, 256)), dim3(256), 0, s, T, E, k, token_ids,
                      topk_idx, topk_w);
}

cudaError_t launch_router_fused(const RouteParams &p, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const dim3 grid((unsigned)ceil_div(p.T, kRouteTokPerCta)), block(256);
    if (p.E <= 8) return launch_pdl(router_fused_kernel<float, 8>, grid, block, 0, s, p);
    if (p.E <= 16) return launch_pdl(router_fused_kernel<float, 16>, grid, block, 0, s, p);
    return launch_pdl(router_fused_kernel<float, 32>, grid, block, 0, s, p);
}

cudaError_t launch_route_logits(const RouteParams &p, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const int E = p.E;
    if (E <= 8) return launch_route_logits_t<8, 1>(p, s);
    if (E <= 16) return launch_route_logits_t<16, 1>(p, s);
    if (E <= 32) return launch_route_logits_t<32, 1>(p, s);
    if (E <= 64) return launch_route_logits_t<32, 2>(p, s);
    if (E <= 128) return launch_route_logits_t<32, 4>(p, s);
    if (E <= 256) return launch_route_logits_t<32, 8>(p, s);
    if (E <= 512) return launch_route_logits_t<32, 16>(p, s);
    return launch_route_logits_t<32, 32>(p, s);
}

cudaError_t launch_router_logits_simt(const RouteParams &p, int dtype, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const dim3 grid((unsigned)ceil_div(p.T, 32), (unsigned)ceil_div(p.E, 32));
    if (dtype == 0)
        return launch_pdl(router_logits_simt_kernel<float>, grid, dim3(256), 0, s, static_cast<const float *>(p.x),
                          static_cast<const float *>(p.w_router), p.logits, p.T, p.E, p.d);
    return launch_pdl(router_logits_simt_kernel<bf16>, grid, dim3(256), 0, s, static_cast<const bf16 *>(p.x),
                      static_cast<const bf16 *>(p.w_router), p.logits, p.T, p.E, p.d);
}

cudaError_t launch_route_reduce(const float *part_prob, const int32_t *part_cnt, int64_t nblk,
                                int E, int64_t T, float *prob_mean, int32_t *counts,
                                cudaStream_t s) {
    return launch_pdl(route_reduce_kernel, dim3((unsigned)E), dim3(256), 0, s, part_prob, part_cnt, nblk, E, T,
                      prob_mean, counts);
}

}  // namespace moe
