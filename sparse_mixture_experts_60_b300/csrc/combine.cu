// Gate-weighted combine back to token order, balance statistics, and the
// aux-loss-free bias update.
//
// Pages: "MoE Training: Mixture of Experts" (Quick Start MoELayer
// output[mask] += score * expert_output; Load Balancing: auxiliary loss
// N sum f_i P_i and router z-loss mean(logsumexp^2)); "Mixture of Experts
// (MoE) From Scratch to DeepSeek V3" (output y = sum Gate_i E_i(x) + x;
// shared experts; bias b_i lowered for an overloaded expert and raised for
// an idle one); "MoE Training Guide" (Monitoring: imbalance, utilisation,
// drop rate).
#include <math.h>
#include <stdint.h>

#include "moe_b300.h"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// One warp per token; each lane owns V consecutive output columns per step.
//   out = sum_j w_j * y[inv_j]  (j ascending, dropped slots skipped)
//         + z (shared expert) + x (residual), in fp32, stored in dtype.
// PRE: the rows already hold w_j * y (+ x for the token's first kept slot,
// CombinePrep): out = sum_j y[inv_j] + z, + x only if no slot was kept.
template <bool BF16, bool PRE = false>
__global__ void __launch_bounds__(256) combine_kernel(int64_t T, int d, int k, const float *__restrict__ y,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ topk_w,
                                                      const float *__restrict__ z, const void *__restrict__ x,
                                                      void *__restrict__ out) {
    PDL_ENTER();
    constexpr int V = BF16 ? 8 : 4;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int my_r = lane < k ? inv[t * k + lane] : -1;
    const float my_w = (!PRE && lane < k) ? topk_w[t * k + lane] : 1.0f;
    int rows[kMaxTopK];
    float wts[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        rows[j] = __shfl_sync(kFull, my_r, j);
        wts[j] = __shfl_sync(kFull, my_w, j);
    }
    // with prepared rows x is already in the first kept row
    if (PRE && __any_sync(kFull, lane < k && my_r >= 0)) x = nullptr;
    const int nchunk = d / V;
    for (int c = lane; c < nchunk; c += 32) {
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j < k && rows[j] >= 0) {
                const float4 *src = reinterpret_cast<const float4 *>(y + (int64_t)rows[j] * d) + c * (V / 4);
#pragma unroll
                for (int h = 0; h < V / 4; ++h) {
                    const float4 u = __ldg(src + h);
                    if (PRE) {
                        acc[4 * h + 0] += u.x;
                        acc[4 * h + 1] += u.y;
                        acc[4 * h + 2] += u.z;
                        acc[4 * h + 3] += u.w;
                    } else {
                        acc[4 * h + 0] = fmaf(wts[j], u.x, acc[4 * h + 0]);
                        acc[4 * h + 1] = fmaf(wts[j], u.y, acc[4 * h + 1]);
                        acc[4 * h + 2] = fmaf(wts[j], u.z, acc[4 * h + 2]);
                        acc[4 * h + 3] = fmaf(wts[j], u.w, acc[4 * h + 3]);
                    }
                }
            }
        }
        if (z) {
            const float4 *src = reinterpret_cast<const float4 *>(z + t * d) + c * (V / 4);
#pragma unroll
            for (int h = 0; h < V / 4; ++h) {
                const float4 u = __ldg(src + h);
                acc[4 * h + 0] += u.x;
                acc[4 * h + 1] += u.y;
                acc[4 * h + 2] += u.z;
                acc[4 * h + 3] += u.w;
            }
        }
        if (BF16) {
            if (x) {
                const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(x) + t * d) + c);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    acc[2 * h] += __uint_as_float(w[h] << 16);
                    acc[2 * h + 1] += __uint_as_float(w[h] & 0xffff0000u);
                }
            }
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * h], acc[2 * h + 1]);
                o[h] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            reinterpret_cast<uint4 *>(static_cast<bf16 *>(out) + t * d)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            if (x) {
                const float4 u = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) + t * d) + c);
                acc[0] += u.x;
                acc[1] += u.y;
                acc[2] += u.z;
                acc[3] += u.w;
            }
            reinterpret_cast<float4 *>(static_cast<float *>(out) + t * d)[c] =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
    }
}

// The combine of prepared rows (CombinePrep) for k = KC in {1, 2, 4, 8},
// bf16 layers: warp per token, each lane H 8-column chunks per step (two for
// k <= 2, columns c and c + 256; one for larger k, to bound the registers)
// with every row load of the step issued before the first add; out = sum_j y[inv_j] (j ascending) + z, + x only if no slot of
// the token was kept, as combine_kernel<true, true>.
template <int KC, int H = (KC <= 2 ? 2 : 1)>
__global__ void __launch_bounds__(256) combine_pre_kernel(int64_t T, int d, const float *__restrict__ y,
                                                          const int32_t *__restrict__ inv,
                                                          const float *__restrict__ z, const bf16 *__restrict__ x,
                                                          bf16 *__restrict__ out) {
    PDL_ENTER();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int my_r = lane < KC ? __ldg(inv + t * KC + lane) : -1;
    int rows[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) rows[j] = __shfl_sync(kFull, my_r, j);
    if (__any_sync(kFull, lane < KC && my_r >= 0)) x = nullptr;
    const int nchunk = d / 8;
    for (int c0 = lane; c0 < nchunk; c0 += 32 * H) {
        float4 u[KC][H][2];
#pragma unroll
        for (int j = 0; j < KC; ++j)
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const int c = c0 + 32 * h;
                const bool ok = rows[j] >= 0 && c < nchunk;
                const float4 *src = reinterpret_cast<const float4 *>(y + (int64_t)(ok ? rows[j] : 0) * d) + 2 * c;
                u[j][h][0] = ok ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
                u[j][h][1] = ok ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        float4 zz[H][2];
        uint4 xx[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const int c = c0 + 32 * h;
            const bool ok = c < nchunk;
            zz[h][0] = zz[h][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            xx[h] = make_uint4(0, 0, 0, 0);
            if (ok && z) {
                zz[h][0] = __ldg(reinterpret_cast<const float4 *>(z + t * d) + 2 * c);
                zz[h][1] = __ldg(reinterpret_cast<const float4 *>(z + t * d) + 2 * c + 1);
            }
            if (ok && x) xx[h] = __ldg(reinterpret_cast<const uint4 *>(x + t * d) + c);
        }
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const int c = c0 + 32 * h;
            if (c >= nchunk) continue;
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                if (rows[j] < 0) continue;
                const float v[8] = {u[j][h][0].x, u[j][h][0].y, u[j][h][0].z, u[j][h][0].w,
                                    u[j][h][1].x, u[j][h][1].y, u[j][h][1].z, u[j][h][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += v[i];
            }
            if (z) {
                const float v[8] = {zz[h][0].x, zz[h][0].y, zz[h][0].z, zz[h][0].w,
                                    zz[h][1].x, zz[h][1].y, zz[h][1].z, zz[h][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += v[i];
            }
            if (x) {
                const uint32_t w[4] = {xx[h].x, xx[h].y, xx[h].z, xx[h].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += __uint_as_float(w[q] << 16);
                    acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
                }
            }
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
                o[q] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            reinterpret_cast<uint4 *>(out + t * d)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Combine for more than kMaxTopK slots per token (expert-choice routing on
// many experts).  Warp per token: the token's kept (row, gate) pairs are
// first compacted into a per-warp shared list in slot order (ballots over 32
// slots at a time), then summed in that order like the narrow kernel.
template <bool BF16>
__global__ void __launch_bounds__(256) combine_wide_kernel(int64_t T, int d, int k, const float *__restrict__ y,
                                                           const int32_t *__restrict__ inv,
                                                           const float *__restrict__ topk_w,
                                                           const float *__restrict__ z, const void *__restrict__ x,
                                                           void *__restrict__ out) {
    PDL_ENTER();
    extern __shared__ int wlist[];                       // [8 warps][k] rows, then [8][k] gates
    constexpr int V = BF16 ? 8 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * 8 + warp;
    if (t >= T) return;
    int *rows = wlist + warp * k;
    float *wts = reinterpret_cast<float *>(wlist + 8 * k) + warp * k;
    int n = 0;
    for (int j0 = 0; j0 < k; j0 += 32) {
        const int j = j0 + lane;
        const int r = j < k ? __ldg(inv + t * k + j) : -1;
        const unsigned b = __ballot_sync(kFull, r >= 0);
        if (r >= 0) {
            const int pos = n + __popc(b & ((1u << lane) - 1u));
            rows[pos] = r;
            wts[pos] = __ldg(topk_w + t * k + j);
        }
        n += __popc(b);
    }
    __syncwarp();
    for (int c = lane; c < d / V; c += 32) {
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.0f;
        for (int i = 0; i < n; ++i) {
            const float4 *src = reinterpret_cast<const float4 *>(y + (int64_t)rows[i] * d) + c * (V / 4);
            const float wv = wts[i];
#pragma unroll
            for (int h = 0; h < V / 4; ++h) {
                const float4 u = __ldg(src + h);
                acc[4 * h + 0] = fmaf(wv, u.x, acc[4 * h + 0]);
                acc[4 * h + 1] = fmaf(wv, u.y, acc[4 * h + 1]);
                acc[4 * h + 2] = fmaf(wv, u.z, acc[4 * h + 2]);
                acc[4 * h + 3] = fmaf(wv, u.w, acc[4 * h + 3]);
            }
        }
        if (z) {
            const float4 *src = reinterpret_cast<const float4 *>(z + t * d) + c * (V / 4);
#pragma unroll
            for (int h = 0; h < V / 4; ++h) {
                const float4 u = __ldg(src + h);
                acc[4 * h + 0] += u.x;
                acc[4 * h + 1] += u.y;
                acc[4 * h + 2] += u.z;
                acc[4 * h + 3] += u.w;
            }
        }
        if (BF16) {
            if (x) {
                const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(x) + t * d) + c);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    acc[2 * h] += __uint_as_float(w[h] << 16);
                    acc[2 * h + 1] += __uint_as_float(w[h] & 0xffff0000u);
                }
            }
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * h], acc[2 * h + 1]);
                o[h] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            reinterpret_cast<uint4 *>(static_cast<bf16 *>(out) + t * d)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            if (x) {
                const float4 u = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) + t * d) + c);
                acc[0] += u.x;
                acc[1] += u.y;
                acc[2] += u.z;
                acc[3] += u.w;
            }
            reinterpret_cast<float4 *>(static_cast<float *>(out) + t * d)[c] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
    }
}

template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

struct AddF { __device__ float operator()(float a, float b) const { return a + b; } };
struct AddL { __device__ long long operator()(long long a, long long b) const { return a + b; } };
struct MaxL { __device__ long long operator()(long long a, long long b) const { return a > b ? a : b; } };
struct MinL { __device__ long long operator()(long long a, long long b) const { return a < b ? a : b; } };

// Single CTA, fp32 throughout, deterministic and free of fp64: per-thread
// strided sums (Kahan-compensated over lse), xor butterflies inside warps,
// then one shared-memory round folded by thread 0 in warp order.  P and z
// come from the router's per-block partials in the layer forward (a warp
// per expert over the blocks), from prob_mean / lse in moe_stats.
__global__ void __launch_bounds__(512) stats_kernel(StatsParams p) {
    PDL_ENTER();
    __shared__ float sP[kMaxExperts];
    __shared__ float red_f[32][2];
    __shared__ long long red_l[32][5];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t S = p.T * p.k;
    const bool parts = p.part_prob != nullptr;
    const bool have_p = parts || p.prob_mean;
    const bool have_z = (parts && p.part_z) || p.lse;
    float z = 0.0f;
    if (parts && p.part_z) {
        for (int64_t b = threadIdx.x; b < p.nblk; b += blockDim.x) z += p.part_z[b];
    } else if (p.lse) {
        float zc = 0.0f;
        for (int64_t i = threadIdx.x; i < p.T; i += blockDim.x) {
            const float v = p.lse[i] * p.lse[i] - zc;
            const float t = z + v;
            zc = (t - z) - v;
            z = t;
        }
    }
    if (parts) {
        for (int e = warp; e < p.E; e += (int)(blockDim.x >> 5)) {
            float acc = 0.0f;
            for (int64_t b = lane; b < p.nblk; b += 32) acc += p.part_prob[(int64_t)e * p.nblk + b];
            acc = warp_reduce(acc, AddF());
            if (lane == 0) {
                const float P = p.T > 0 ? acc / (float)p.T : 0.0f;
                sP[e] = P;
                if (p.prob_out) p.prob_out[e] = P;
            }
        }
    } else if (p.prob_mean) {
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) sP[e] = p.prob_mean[e];
    }
    __syncthreads();
    float aux = 0.0f;
    long long dropped = 0, used = 0, kept_tot = 0, kmax = 0, kmin = 0x7fffffffffffffffLL;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        const float f = S > 0 ? (float)p.counts[e] / (float)S : 0.0f;
        if (p.f) p.f[e] = f;
        if (have_p) aux += f * sP[e];
        dropped += p.counts[e] - p.kept[e];
        used += p.kept[e] > 0;
        kept_tot += p.kept[e];
        kmax = p.kept[e] > kmax ? p.kept[e] : kmax;
        kmin = p.kept[e] < kmin ? p.kept[e] : kmin;
    }
    z = warp_reduce(z, AddF());
    aux = warp_reduce(aux, AddF());
    dropped = warp_reduce(dropped, AddL());
    used = warp_reduce(used, AddL());
    kept_tot = warp_reduce(kept_tot, AddL());
    kmax = warp_reduce(kmax, MaxL());
    kmin = warp_reduce(kmin, MinL());
    if (lane == 0) {
        red_f[warp][0] = z;
        red_f[warp][1] = aux;
        red_l[warp][0] = dropped;
        red_l[warp][1] = used;
        red_l[warp][2] = kept_tot;
        red_l[warp][3] = kmax;
        red_l[warp][4] = kmin;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        for (int w = 1; w < nw; ++w) {
            z += red_f[w][0];
            aux += red_f[w][1];
            dropped += red_l[w][0];
            used += red_l[w][1];
            kept_tot += red_l[w][2];
            kmax = red_l[w][3] > kmax ? red_l[w][3] : kmax;
            kmin = red_l[w][4] < kmin ? red_l[w][4] : kmin;
        }
        moe_stats_t st;
        // without router probabilities (routing given by the caller) the
        // balance losses are undefined: NaN
        st.aux_loss = have_p ? (float)p.E * aux : __int_as_float(0x7fc00000);
        st.z_loss = !have_z ? __int_as_float(0x7fc00000) : (p.T > 0 ? z / (float)p.T : 0.0f);
        st.imbalance = kmin > 0 ? (float)kmax / (float)kmin : INFINITY;
        st.utilization = (float)used / (float)p.E;
        st.drop_rate = S > 0 ? (float)dropped / (float)S : 0.0f;
        st.dropped = (int32_t)dropped;
        st.capacity = p.drop ? (int32_t)p.cap : -1;
        st.total_kept = (int32_t)kept_tot;
        *static_cast<moe_stats_t *>(p.stats) = st;
    }
}

__global__ void bias_update_kernel(int64_t S, int E, const int32_t *counts, float *b, float gamma) {
    PDL_ENTER();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const long long diff = (long long)S - (long long)E * counts[e];  // sign of S/E - counts_e
    const float sg = diff > 0 ? 1.0f : (diff < 0 ? -1.0f : 0.0f);
    b[e] = __fadd_rn(b[e], __fmul_rn(gamma, sg));
}

}  // namespace

cudaError_t launch_combine(int64_t T, int d, int k, int dtype, const float *y_perm, const int32_t *inv,
                           const float *topk_w, const float *shared_out, const void *x_res, void *out,
                           cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const unsigned grid = (unsigned)ceil_div(T, 8);
    if (k > kMaxTopK) {
        const size_t smem = (size_t)16 * k * sizeof(int);
        auto kern = dtype == 1 ? combine_wide_kernel<true> : combine_wide_kernel<false>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(kern, dim3(grid), dim3(256), smem, s, T, d, k, y_perm, inv, topk_w, shared_out, x_res,
                          out);
    }
    auto kern = dtype == 1 ? combine_kernel<true> : combine_kernel<false>;
    return launch_pdl(kern, dim3(grid), dim3(256), 0, s, T, d, k, y_perm, inv, topk_w, shared_out, x_res, out);
}

cudaError_t launch_combine_prepped(int64_t T, int d, int k, int dtype, const float *y_perm, const int32_t *inv,
                                   const float *shared_out, const void *x_res, void *out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (k > kMaxTopK) return cudaErrorInvalidValue;
    if (dtype == 1 && (k == 1 || k == 2 || k == 4 || k == 8)) {
        auto kern = k == 1 ? combine_pre_kernel<1>
                           : (k == 2 ? combine_pre_kernel<2> : (k == 4 ? combine_pre_kernel<4> : combine_pre_kernel<8>));
        return launch_pdl(kern, dim3((unsigned)ceil_div(T, 8)), dim3(256), 0, s, T, d, y_perm, inv, shared_out,
                          static_cast<const bf16 *>(x_res), static_cast<bf16 *>(out));
    }
    auto kern = dtype == 1 ? combine_kernel<true, true> : combine_kernel<false, true>;
    return launch_pdl(kern, dim3((unsigned)ceil_div(T, 8)), dim3(256), 0, s, T, d, k, y_perm, inv,
                      static_cast<const float *>(nullptr), shared_out, x_res, out);
}

cudaError_t launch_stats(const StatsParams &p, cudaStream_t s) {
    return launch_pdl(stats_kernel, dim3(1), dim3(512), 0, s, p);
}

cudaError_t launch_bias_update(int64_t T, int E, int k, const int32_t *counts, float *bias, float gamma,
                               cudaStream_t s) {
    return launch_pdl(bias_update_kernel, dim3((unsigned)ceil_div(E, 256)), dim3(256), 0, s, T * k, E, counts, bias,
                      gamma);
}

}  // namespace moe
