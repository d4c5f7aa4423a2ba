// Backward of the layer, the kernels around the tensor-core GEMMs:
//   combine backward  dy = gate * dout into the expert rows, dgate = <dout, y>
//   router backward   dlogits from the gate Jacobian, L_aux and z-loss
//   dx assembly       sum of the expert rows' dx, residual, shared expert,
//                     and the router term dlogits W_r
//   router weights    dW_r = dlogits^T x, db_r (two-pass, fixed order)
//   packed transpose  dlogits and x, K-major with the tokens padded to a
//                     multiple of 64 (zeros): the operands of a wide
//                     router's dW_r GEMM
//   bias gradients    per-expert sums of da and dy over their rows
//
// No page prints a backward; the objective is the one the "MoE Training:
// Mixture of Experts" page trains, the layer output plus the auxiliary
// (load-balancing) loss and the router z-loss, and every kernel below is a
// term of its chain rule.
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        f[2 * h] = __uint_as_float(w[h] << 16);
        f[2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * h], f[2 * h + 1]);
        w[h] = *reinterpret_cast<const uint32_t *>(&b2);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Warp per token.  For every kept slot j (row = inv[t,j]):
//   dy[row] = bf16(gate * dout_t),  dgate[t,j] = sum_n dout_t[n] y[row, n];
// a dropped slot gets dgate = 0.  d % 8 == 0 (bf16 vectors of 8).
__global__ void __launch_bounds__(256) combine_bwd_kernel(int64_t T, int d, int k, const bf16 *__restrict__ dout,
                                                          const float *__restrict__ topk_w,
                                                          const int32_t *__restrict__ inv,
                                                          const float *__restrict__ y, bf16 *__restrict__ dy,
                                                          float *__restrict__ dgate) {
    PDL_ENTER();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint4 *go = reinterpret_cast<const uint4 *>(dout + t * d);
    const int nv = d / 8;
    for (int j = 0; j < k; ++j) {
        const int32_t row = __ldg(inv + t * k + j);
        if (row < 0) {
            if (lane == 0) dgate[t * k + j] = 0.0f;
            continue;
        }
        const float g = __ldg(topk_w + t * k + j);
        const float4 *yr = reinterpret_cast<const float4 *>(y + (int64_t)row * d);
        uint4 *dyr = reinterpret_cast<uint4 *>(dy + (int64_t)row * d);
        float dot = 0.0f;
        for (int c = lane; c < nv; c += 32) {
            float o[8], gy[8];
            unpack8(__ldg(go + c), o);
            const float4 y0 = __ldg(yr + 2 * c), y1 = __ldg(yr + 2 * c + 1);
            const float yy[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                dot = fmaf(o[i], yy[i], dot);
                gy[i] = g * o[i];
            }
            dyr[c] = pack8(gy);
        }
        dot = warp_sum(dot);
        if (lane == 0) dgate[t * k + j] = dot;
    }
}

// Warp per token: dlogits[t, :] (fp32).  p = softmax(l_t); the gate
// gradient goes through the forward's gate function (softmax or sigmoid,
// renormalised over the chosen experts or not), then the auxiliary loss
// (f_e = counts_e / (T k) held fixed) and the z-loss terms are added.
// Per-warp shared scratch: dg[E] (gate gradient per chosen expert) and
// sel[E] (1 for a chosen expert).  dl_hi / dl_lo (optional): dl split into
// two bf16 numbers (hi = bf16(dl), lo = bf16(dl - hi)), the operands of the
// router's tensor-core GEMMs on wide routers (hi + lo keeps ~16 bits).
__global__ void __launch_bounds__(256) router_bwd_kernel(int64_t T, int E, int k, int score_fn, int renormalize,
                                                         const float *__restrict__ logits,
                                                         const int32_t *__restrict__ topk_idx,
                                                         const float *__restrict__ dgate,
                                                         const int32_t *__restrict__ counts, float aux_coef,
                                                         float z_coef, float *__restrict__ dl,
                                                         bf16 *__restrict__ dl_hi, bf16 *__restrict__ dl_lo) {
    PDL_ENTER();
    extern __shared__ float sh[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float *dg = sh + warp * 2 * E;
    float *sel = dg + E;
    const int64_t t = (int64_t)blockIdx.x * 8 + warp;
    if (t >= T) return;
    const float *l = logits + t * E;
    for (int e = lane; e < E; e += 32) {
        dg[e] = 0.0f;
        sel[e] = 0.0f;
    }
    __syncwarp();
    if (lane < k) {
        const int e = __ldg(topk_idx + t * k + lane);
        dg[e] = __ldg(dgate + t * k + lane);
        sel[e] = 1.0f;
    }
    __syncwarp();
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, __ldg(l + e));
    m = warp_max(m);
    float s = 0.0f;
    for (int e = lane; e < E; e += 32) s += expf(__ldg(l + e) - m);
    s = warp_sum(s);
    const float lse = m + logf(s);
    const float inv_tk = 1.0f / (float)(T * k);
    // gate values v (softmax p or sigmoid s) summed over the chosen experts;
    // renormalised gates w = v / tot, then sum_j w_j dg_j (raw: sum_j v_j dg_j).
    // Written as w (dg - sum w dg), a top-1 renormalised gate (w = 1
    // exactly) passes exactly zero.
    float tot = 0.0f, fp = 0.0f;
    for (int e = lane; e < E; e += 32) {
        const float le = __ldg(l + e);
        const float p = expf(le - lse);
        tot += sel[e] * (score_fn == 0 ? p : 1.0f / (1.0f + expf(-le)));
        fp += (float)__ldg(counts + e) * inv_tk * p;
    }
    tot = warp_sum(tot);
    fp = warp_sum(fp);
    float wdg = 0.0f;
    for (int e = lane; e < E; e += 32) {
        const float le = __ldg(l + e);
        const float v = score_fn == 0 ? expf(le - lse) : 1.0f / (1.0f + expf(-le));
        wdg += sel[e] * (renormalize ? v / tot : v) * dg[e];
    }
    wdg = warp_sum(wdg);
    const float aux_s = aux_coef * (float)E / (float)T, z_s = z_coef * 2.0f / (float)T * lse;
    for (int e = lane; e < E; e += 32) {
        const float le = __ldg(l + e);
        const float p = expf(le - lse);
        float g;
        if (score_fn == 0) {
            g = renormalize ? sel[e] * (p / tot) * (dg[e] - wdg) : p * (sel[e] * dg[e] - wdg);
        } else {
            const float sg = 1.0f / (1.0f + expf(-le));
            g = sel[e] * sg * (1.0f - sg) * (renormalize ? (dg[e] - wdg) / tot : dg[e]);
        }
        g += aux_s * p * ((float)__ldg(counts + e) * inv_tk - fp);
        g += z_s * p;
        dl[t * E + e] = g;
        if (dl_hi) {
            const bf16 hi = __float2bfloat16(g);
            dl_hi[t * E + e] = hi;
            dl_lo[t * E + e] = __float2bfloat16(g - __bfloat162float(hi));
        }
    }
}

// Warp per token, 8 columns per lane step:
//   dx[t] = sum_j dx_perm[inv[t,j]] + dout_t (residual) + dxs[t] (shared)
//           + sum_e dl[t,e] W_r[e, :]   (or dxr[t], that product from the
//           tensor cores on wide routers)
__global__ void __launch_bounds__(256) dx_assemble_kernel(int64_t T, int d, int k, int E,
                                                          const float *__restrict__ dx_perm,
                                                          const int32_t *__restrict__ inv,
                                                          const bf16 *__restrict__ dout, int residual,
                                                          const float *__restrict__ dxs,
                                                          const float *__restrict__ dl,
                                                          const bf16 *__restrict__ w_router,
                                                          const float *__restrict__ dxr, float *__restrict__ dx) {
    PDL_ENTER();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int nv = d / 8;
    for (int c = lane; c < nv; c += 32) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int32_t row = __ldg(inv + t * k + j);
            if (row < 0) continue;
            const float4 *p = reinterpret_cast<const float4 *>(dx_perm + (int64_t)row * d) + 2 * c;
            const float4 a = __ldg(p), b = __ldg(p + 1);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        if (residual) {
            float o[8];
            unpack8(__ldg(reinterpret_cast<const uint4 *>(dout + t * d) + c), o);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += o[i];
        }
        if (dxs) {
            const float4 *p = reinterpret_cast<const float4 *>(dxs + t * d) + 2 * c;
            const float4 a = __ldg(p), b = __ldg(p + 1);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        if (dxr) {
            const float4 *p = reinterpret_cast<const float4 *>(dxr + t * d) + 2 * c;
            const float4 a = __ldg(p), b = __ldg(p + 1);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        } else {
            for (int e = 0; e < E; ++e) {
                const float g = __ldg(dl + t * E + e);
                float wv[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(w_router + (int64_t)e * d) + c), wv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, wv[i], acc[i]);
            }
        }
        float4 *o = reinterpret_cast<float4 *>(dx + t * d) + 2 * c;
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// Router weight gradient, pass 1: CTA (column block of 128, token chunk)
// accumulates sum_t dl[t, e] x[t, col] for 32 experts at a time into
// part[chunk][e][col].
constexpr int kRwCols = 128;
constexpr int kRwChunk = 512;
template <int EP>
__global__ void __launch_bounds__(kRwCols) router_wgrad_partial_kernel(int64_t T, int d, int E,
                                                                      const float *__restrict__ dl,
                                                                      const bf16 *__restrict__ x,
                                                                      float *__restrict__ part) {
    PDL_ENTER();
    __shared__ float sdl[32][EP + 1];
    const int col = blockIdx.x * kRwCols + threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.y * kRwChunk;
    const int64_t t1 = t0 + kRwChunk < T ? t0 + kRwChunk : T;
    for (int e0 = 0; e0 < E; e0 += EP) {
        float acc[EP];
#pragma unroll
        for (int i = 0; i < EP; ++i) acc[i] = 0.0f;
        for (int64_t tb = t0; tb < t1; tb += 32) {
            __syncthreads();
            for (int i = threadIdx.x; i < 32 * EP; i += kRwCols) {
                const int tt = i / EP, ee = i % EP;
                sdl[tt][ee] = (tb + tt < t1 && e0 + ee < E) ? __ldg(dl + (tb + tt) * E + e0 + ee) : 0.0f;
            }
            __syncthreads();
            const int nt = (int)(t1 - tb < 32 ? t1 - tb : 32);
            for (int tt = 0; tt < nt; ++tt) {
                const float xv = col < d ? __bfloat162float(x[(tb + tt) * d + col]) : 0.0f;
#pragma unroll
                for (int ee = 0; ee < EP; ++ee) acc[ee] = fmaf(sdl[tt][ee], xv, acc[ee]);
            }
        }
        if (col < d) {
#pragma unroll
            for (int ee = 0; ee < EP; ++ee)
                if (e0 + ee < E) part[((int64_t)blockIdx.y * E + e0 + ee) * d + col] = acc[ee];
        }
    }
}

// Pass 2: dW_r[e, col] = sum over chunks in order; db_r[e] = sum_t dl[t, e]
// (thread per column, block per expert).
__global__ void __launch_bounds__(256) router_wgrad_reduce_kernel(int64_t T, int d, int E, int nchunk,
                                                                 const float *__restrict__ part,
                                                                 const float *__restrict__ dl,
                                                                 float *__restrict__ dw, float *__restrict__ db) {
    PDL_ENTER();
    __shared__ float red[256];
    const int e = blockIdx.y;
    for (int col = blockIdx.x * 256 + threadIdx.x; col < d && dw; col += gridDim.x * 256) {
        float s = 0.0f;
        for (int c = 0; c < nchunk; ++c) s += part[((int64_t)c * E + e) * d + col];
        dw[(int64_t)e * d + col] = s;
    }
    if (db && blockIdx.x == 0) {
        float s = 0.0f;
        for (int64_t t = threadIdx.x; t < T; t += 256) s += dl[t * E + e];
        red[threadIdx.x] = s;
        __syncthreads();
        for (int st = 128; st > 0; st >>= 1) {
            if (threadIdx.x < st) red[threadIdx.x] += red[threadIdx.x + st];
            __syncthreads();
        }
        if (threadIdx.x == 0) db[e] = red[0];
    }
}

// 64 x 64 bf16 tile transpose through shared memory with 16-byte global
// accesses on both sides: 256 threads each load two 8-element row vectors
// (rows past `nrows`, columns past `ncols` read as zeros), then each
// gathers two 8-row column vectors.  Rows are 128 bytes, their eight 16-byte
// chunks XOR-swizzled by (row / 8) mod 8: a warp's row writes cover whole
// rows, and the eight threads of a column gather (rows 8j .. 8j+7, j = 0..7)
// read eight different chunks, so neither side has bank conflicts.
__device__ __forceinline__ int swz(int r, int c) { return (((c >> 3) ^ ((r >> 3) & 7)) << 3) | (c & 7); }
template <typename SrcRow>
__device__ __forceinline__ void tile_in(bf16 (*tile)[64], SrcRow src_row, int nrows, int ncols) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int v = threadIdx.x + h * 256;          // 512 vectors: row v / 8, columns 8 (v % 8) ..
        const int r = v >> 3, c8 = (v & 7) * 8;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (r < nrows && c8 < ncols) u = __ldg(reinterpret_cast<const uint4 *>(src_row(r) + c8));
        *reinterpret_cast<uint4 *>(&tile[r][swz(r, c8)]) = u;
    }
}
__device__ __forceinline__ uint4 tile_col8(bf16 (*tile)[64], int c, int r8) {
    uint32_t w[4];
    const int pc = swz(r8, c);                         // rows r8 .. r8+7 share the swizzle
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint32_t lo = __bfloat16_as_ushort(tile[r8 + 2 * h][pc]);
        const uint32_t hi = __bfloat16_as_ushort(tile[r8 + 2 * h + 1][pc]);
        w[h] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Packed transpose of grouped rows: out[c][pad[g] + i] = in[off[g] + i][c]
// for i < rows_g, zero for rows_g <= i < pad[g+1] - pad[g].  Every pad[g]
// is a multiple of 64, so a 64-column output tile belongs to one group.
// off == nullptr: a single group of `rows` rows.  cols, ld_in multiples of 8.
__global__ void __launch_bounds__(256) transpose_pack_kernel(const bf16 *__restrict__ in, int ld_in, int cols,
                                                             const int32_t *__restrict__ off,
                                                             const int32_t *__restrict__ pad, int G, int rows,
                                                             bf16 *__restrict__ out, int64_t ld_out) {
    PDL_ENTER();
    __shared__ __align__(16) bf16 tile[64][64];
    const int p0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    const int total = pad[G];
    if (p0 >= total) return;
    int g = 0;
    if (off) {
        int lo = 0, hi = G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pad[mid] <= p0) lo = mid;
            else hi = mid - 1;
        }
        g = lo;
    }
    const int gbeg = off ? off[g] : 0, gend = off ? off[g + 1] : rows;
    const int r0 = gbeg + (p0 - pad[g]);                  // first source row of the tile
    const int nr = gend - r0 < 64 ? (gend - r0 > 0 ? gend - r0 : 0) : 64;
    const int nc = cols - c0 < 64 ? cols - c0 : 64;
    tile_in(tile, [&](int r) { return in + (int64_t)(r0 + r) * ld_in + c0; }, nr, nc);
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int v = threadIdx.x + h * 256;
        const int c = v >> 3, r8 = (v & 7) * 8;
        if (c < nc) *reinterpret_cast<uint4 *>(out + (int64_t)(c0 + c) * ld_out + p0 + r8) = tile_col8(tile, c, r8);
    }
}

// pad[0] = 0, pad[g+1] = pad[g] + roundup(off[g+1] - off[g], 64); one CTA,
// fixed-order block scan.  off == nullptr: one group of `rows` rows.
__global__ void __launch_bounds__(1024) pad_offsets_kernel(const int32_t *__restrict__ off, int G, int rows,
                                                           int32_t *__restrict__ pad) {
    PDL_ENTER();
    __shared__ int wsum[32];
    __shared__ int carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        pad[0] = 0;
    }
    __syncthreads();
    for (int b = 0; b < G; b += blockDim.x) {
        const int g = b + threadIdx.x;
        int v = 0;
        if (g < G) {
            const int n = off ? off[g + 1] - off[g] : rows;
            v = (n + 63) / 64 * 64;
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += u;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(kFull, w, o);
                if (lane >= o) w += u;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int incl = carry + (warp > 0 ? wsum[warp - 1] : 0) + x;
        if (g < G) pad[g + 1] = incl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
}

// Per-group column sums of a row-major bf16 matrix (bias gradients):
// out[g][c] = sum over rows off[g] .. off[g+1]-1 of in[r][c], thread per
// column, rows in order (deterministic).
__global__ void __launch_bounds__(256) group_colsum_kernel(const bf16 *__restrict__ in, int64_t ld,
                                                           const int32_t *__restrict__ off, int C,
                                                           float *__restrict__ out) {
    PDL_ENTER();
    const int g = blockIdx.y;
    const int c = blockIdx.x * 256 + threadIdx.x;
    if (c >= C) return;
    const int r0 = off[g], r1 = off[g + 1];
    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
    int r = r0;
    for (; r + 3 < r1; r += 4) {
        s0 += __bfloat162float(in[(int64_t)r * ld + c]);
        s1 += __bfloat162float(in[(int64_t)(r + 1) * ld + c]);
        s2 += __bfloat162float(in[(int64_t)(r + 2) * ld + c]);
        s3 += __bfloat162float(in[(int64_t)(r + 3) * ld + c]);
    }
    for (; r < r1; ++r) s0 += __bfloat162float(in[(int64_t)r * ld + c]);
    out[(int64_t)g * C + c] = (s0 + s1) + (s2 + s3);
}

__global__ void fill_range_kernel(int32_t *seg, int n) {
    PDL_ENTER();
    seg[0] = 0;
    seg[1] = n;
}

}  // namespace

cudaError_t launch_group_colsum(const bf16 *in, int64_t ld, const int32_t *off, int G, int C, float *out,
                                cudaStream_t s) {
    if ((int64_t)G * C == 0) return cudaSuccess;
    return launch_pdl(group_colsum_kernel, dim3((unsigned)ceil_div(C, 256), (unsigned)G), dim3(256), 0, s, in, ld,
                      off, C, out);
}

cudaError_t launch_fill_range(int32_t *seg, int n, cudaStream_t s) {
    return launch_pdl(fill_range_kernel, dim3(1), dim3(1), 0, s, seg, n);
}

cudaError_t launch_combine_bwd(int64_t T, int d, int k, const bf16 *dout, const float *topk_w, const int32_t *inv,
                               const float *y, bf16 *dy, float *dgate, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(combine_bwd_kernel, dim3((unsigned)ceil_div(T, 8)), dim3(256), 0, s, T, d, k, dout, topk_w,
                      inv, y, dy, dgate);
}

cudaError_t launch_router_bwd(int64_t T, int E, int k, int score_fn, int renormalize, const float *logits,
                              const int32_t *topk_idx, const float *dgate, const int32_t *counts, float aux_coef,
                              float z_coef, float *dl, bf16 *dl_hi, bf16 *dl_lo, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)8 * 2 * E * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(router_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(router_bwd_kernel, dim3((unsigned)ceil_div(T, 8)), dim3(256), smem, s, T, E, k, score_fn,
                      renormalize, logits, topk_idx, dgate, counts, aux_coef, z_coef, dl, dl_hi, dl_lo);
}

cudaError_t launch_dx_assemble(int64_t T, int d, int k, int E, const float *dx_perm, const int32_t *inv,
                               const bf16 *dout, int residual, const float *dxs, const float *dl,
                               const bf16 *w_router, const float *dxr, float *dx, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(dx_assemble_kernel, dim3((unsigned)ceil_div(T, 8)), dim3(256), 0, s, T, d, k, E, dx_perm,
                      inv, dout, residual, dxs, dl, w_router, dxr, dx);
}

int64_t router_wgrad_chunks(int64_t T) { return ceil_div(T, kRwChunk); }

cudaError_t launch_router_wgrad(int64_t T, int d, int E, const float *dl, const bf16 *x, float *part, float *dw,
                                float *db, cudaStream_t s) {
    if (T == 0) {
        if (dw) {
            const cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)E * d * sizeof(float), s);
            if (e != cudaSuccess) return e;
        }
        return db ? cudaMemsetAsync(db, 0, (size_t)E * sizeof(float), s) : cudaSuccess;
    }
    const int64_t nchunk = router_wgrad_chunks(T);
    cudaError_t e = cudaSuccess;
    if (dw) {
        const dim3 grid((unsigned)ceil_div(d, kRwCols), (unsigned)nchunk);
        if (E <= 8) e = launch_pdl(router_wgrad_partial_kernel<8>, grid, dim3(kRwCols), 0, s, T, d, E, dl, x, part);
        else if (E <= 16)
            e = launch_pdl(router_wgrad_partial_kernel<16>, grid, dim3(kRwCols), 0, s, T, d, E, dl, x, part);
        else e = launch_pdl(router_wgrad_partial_kernel<32>, grid, dim3(kRwCols), 0, s, T, d, E, dl, x, part);
    }
    if (e != cudaSuccess) return e;
    return launch_pdl(router_wgrad_reduce_kernel, dim3((unsigned)ceil_div(d, 256), (unsigned)E), dim3(256), 0, s,
                      T, d, E, (int)nchunk, part, dl, dw, db);
}

cudaError_t launch_transpose_pack(const bf16 *in, int ld_in, int cols, const int32_t *off, const int32_t *pad, int G,
                                  int rows, int64_t max_padded, bf16 *out, int64_t ld_out, cudaStream_t s) {
    if (cols == 0 || max_padded == 0) return cudaSuccess;
    return launch_pdl(transpose_pack_kernel, dim3((unsigned)ceil_div(cols, 64), (unsigned)(max_padded / 64)),
                      dim3(256), 0, s, in, ld_in, cols, off, pad, G, rows, out, ld_out);
}

cudaError_t launch_pad_offsets(const int32_t *off, int G, int rows, int32_t *pad, cudaStream_t s) {
    return launch_pdl(pad_offsets_kernel, dim3(1), dim3(1024), 0, s, off, G, rows, pad);
}

}  // namespace moe
