// Dispatch: per-expert histogram and scan with the capacity clamp, a stable
// rank of every slot within its expert in priority order, the permutation
// and its inverse, and the row copy of x into per-expert segments.
//
// Pages: "MoE Training Guide" (Core MoE Parameters: capacity =
// tokens / num_experts x capacity_factor, min capacity, drop_tokens);
// "Mixture of Experts (MoE) From Scratch to DeepSeek V3" (Token Dropping:
// slots past an expert's buffer are left unprocessed); "MoE Training:
// Mixture of Experts" (Quick Start MoELayer dispatch x_flat[mask], with the
// top-k rank outside and the experts inside, which fixes the priority:
// all rank-0 slots in token order, then rank-1, ...).
//
// Priority index of slot (t, j) is p = j*T + t.  Chunks of kPermChunk
// consecutive priorities are the unit of parallel work.  Layers up to
// kSmallSlots slots dispatch in one CTA (perm_small_kernel); up to a chunk
// table of kTwoPassTable entries in two launches (perm_local_kernel,
// perm_copy_rank_kernel, below); larger ones, and the allocation-free
// entry point, with four:
//   perm_hist  : per-chunk expert histogram                    [nchunk, E]
//   perm_scan  : exclusive scan over chunks per expert (chunk bases),
//                counts, kept = min(counts, C), offsets = scan(kept)
//   perm_rank  : within a chunk, 8 warps x 256 priorities; warp bases from
//                a scan of the warp histograms, then __match_any_sync ranks
//                32 slots at a time in order -> perm, inv
//   perm_copy  : token-major row copy (x read once, written to its k rows)
// Integer work only: the result is unique and deterministic.
#include <stdint.h>

#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPermThreads = 256;
constexpr int kWarpSpan = kPermChunk / (kPermThreads / 32);  // 256 priorities per warp
// two-launch dispatch: chunks of 512, 1024 or 2048 priorities (the
// smallest whose table fits), an eighth of a chunk per warp
constexpr int kLocalChunkMin = 512;

__device__ __forceinline__ int slot_expert(const int32_t *idx, int64_t p, int64_t T, int k, int E,
                                           int64_t S, int64_t *slot_out, int32_t *err) {
    if (p >= S) return -1;
    const int64_t j = p / T, t = p - j * T;
    const int64_t s = t * k + j;
    *slot_out = s;
    const int e = idx[s];
    if (e < 0 || e >= E) {
        if (err) atomicExch(err, 1);  // MOE_ERR_INVALID_ARG
        return -2;
    }
    return e;
}

__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(const int32_t *idx, int64_t T, int k,
                                                                 int E, int32_t *hist, int32_t *err) {
    PDL_ENTER();
    extern __shared__ int h[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int64_t S = T * k;
    const int64_t p0 = (int64_t)blockIdx.x * kPermChunk;
    for (int i = threadIdx.x; i < kPermChunk; i += blockDim.x) {
        int64_t s;
        const int e = slot_expert(idx, p0 + i, T, k, E, S, &s, err);
        if (e >= 0) atomicAdd(&h[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = h[e];
}

// One CTA of 1024 threads (E <= 1024).
__global__ void __launch_bounds__(1024) perm_scan_kernel(const int32_t *hist, int32_t *base,
                                                         int64_t nchunk, int E, int64_t cap,
                                                         int32_t *counts, int32_t *kept,
                                                         int32_t *offsets) {
    PDL_ENTER();
    __shared__ int warp_tot[32];
    const int e = threadIdx.x;
    int kp = 0;
    if (e < E) {
        int run = 0;
        for (int64_t c = 0; c < nchunk; ++c) {
            base[c * E + e] = run;
            run += hist[c * E + e];
        }
        counts[e] = run;
        kp = (int64_t)run < cap ? run : (int)cap;
        kept[e] = kp;
    }
    // exclusive block scan of kept
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int v = kp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += u;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + v - kp;
    if (e < E) offsets[e] = before;
    if (e == E - 1) offsets[E] = before + kp;
}

__global__ void __launch_bounds__(kPermThreads) perm_rank_kernel(const int32_t *idx, int64_t T, int k,
                                                                 int E, int64_t cap,
                                                                 const int32_t *base,
                                                                 const int32_t *offsets,
                                                                 int32_t *perm, int32_t *inv,
                                                                 int32_t *err) {
    PDL_ENTER();
    extern __shared__ int wh[];  // [8][E] warp histograms, then warp running bases
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = kPermThreads / 32;
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wh[i] = 0;
    __syncthreads();
    const int64_t S = T * k;
    const int64_t p0 = (int64_t)blockIdx.x * kPermChunk + (int64_t)warp * kWarpSpan;
    int *my = wh + warp * E;
    // A: warp histogram of its 256 priorities
    for (int g = 0; g < kWarpSpan; g += 32) {
        int64_t s;
        const int e = slot_expert(idx, p0 + g + lane, T, k, E, S, &s, err);
        if (e >= 0) atomicAdd(&my[e], 1);
    }
    __syncthreads();
    // B: exclusive scan over warps, seeded with this chunk's base
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = base[(int64_t)blockIdx.x * E + e];
        for (int w = 0; w < nw; ++w) {
            const int c = wh[w * E + e];
            wh[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    // C: ranks, 32 slots at a time in priority order
    const unsigned lt = (1u << lane) - 1u;
    for (int g = 0; g < kWarpSpan; g += 32) {
        int64_t s = -1;
        const int e = slot_expert(idx, p0 + g + lane, T, k, E, S, &s, err);
        const unsigned peers = __match_any_sync(kFull, e);
        const int rank_in = __popc(peers & lt);
        int rank = 0;
        if (e >= 0) rank = my[e] + rank_in;
        __syncwarp();
        if (e >= 0 && (peers & lt) == 0) my[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            if ((int64_t)rank < cap) {
                const int row = offsets[e] + rank;
                perm[row] = (int32_t)s;
                inv[s] = row;
            } else {
                inv[s] = -1;
            }
        } else if (e == -2) {
            inv[s] = -1;
        }
    }
}

// Dispatch in two launches (layers with nchunk * E <= kTwoPassTable):
//   perm_local_kernel      chunk c (priorities c*lchunk .., lchunk = 512,
//                          1024 or 2048, the smallest whose table fits): the chunk's
//                          expert histogram -> hist[c][E], and every slot's
//                          rank among the chunk's slots of its expert ->
//                          lrank[slot] (8 warps x lchunk/8 priorities, warp bases
//                          from a scan of the warp histograms, match-any
//                          ranks 32 slots at a time)
//   perm_copy_rank_kernel  every CTA first turns the small hist table into
//                          chunk bases, counts, kept and offsets in shared
//                          memory (recomputed per CTA instead of a third
//                          launch); then warp per token: rank = base[chunk of
//                          the slot][e] + lrank[slot], the capacity clamp,
//                          perm / inv, and the row copy of x.
__global__ void __launch_bounds__(kPermThreads) perm_local_kernel(const int32_t *idx, int64_t T, int k, int E,
                                                                  int lchunk, int32_t *hist, int32_t *lrank,
                                                                  int32_t *err) {
    PDL_ENTER();
    extern __shared__ int wh[];          // [8][E] warp histograms, then warp running bases
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nw = kPermThreads / 32;
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wh[i] = 0;
    __syncthreads();
    const int64_t S = T * k;
    const int span = lchunk / nw;
    const int64_t p0 = (int64_t)blockIdx.x * lchunk + (int64_t)warp * span;
    int *my = wh + warp * E;
    for (int g = 0; g < span; g += 32) {
        int64_t sl;
        const int e = slot_expert(idx, p0 + g + lane, T, k, E, S, &sl, err);
        if (e >= 0) atomicAdd(&my[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = wh[w * E + e];
            wh[w * E + e] = run;
            run += c;
        }
        hist[(int64_t)blockIdx.x * E + e] = run;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int g = 0; g < span; g += 32) {
        int64_t sl = -1;
        const int e = slot_expert(idx, p0 + g + lane, T, k, E, S, &sl, nullptr);
        const unsigned peers = __match_any_sync(kFull, e);
        int rank = 0;
        if (e >= 0) rank = my[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && (peers & lt) == 0) my[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) lrank[sl] = rank;
    }
}

__global__ void __launch_bounds__(256) perm_copy_rank_kernel(const uint4 *x, int64_t T, int k, int64_t nvec,
                                                             const int32_t *idx, int E, int64_t cap, int lchunk,
                                                             int64_t nchunk, const int32_t *hist,
                                                             const int32_t *lrank, int32_t *counts, int32_t *kept,
                                                             int32_t *offsets, int32_t *perm, int32_t *inv,
                                                             uint4 *x_perm) {
    PDL_ENTER();
    extern __shared__ int tab[];         // [nchunk][E] chunk bases, then [E + 1] offsets
    __shared__ int scan_s[256];
    int *off_s = tab + nchunk * E;
    const int lane = threadIdx.x & 31;
    const int64_t S = T * k;
    // the chunk table into shared memory in one coalesced pass, then chunk
    // bases (exclusive prefix over chunks) and per-expert totals
    const int64_t ntab = nchunk * E;
    const bool vec = (ntab & 3) == 0 && (reinterpret_cast<uintptr_t>(hist) & 15) == 0;
    if (vec) {
        for (int64_t i = threadIdx.x; i < ntab / 4; i += blockDim.x)
            reinterpret_cast<int4 *>(tab)[i] = __ldg(reinterpret_cast<const int4 *>(hist) + i);
    } else {
        for (int64_t i = threadIdx.x; i < ntab; i += blockDim.x) tab[i] = __ldg(hist + i);
    }
    __syncthreads();
    const int per = (E + 255) / 256;
    const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
    int run_kept = 0;
    for (int e = e0; e < e1; ++e) {
        int run = 0;
        for (int64_t c = 0; c < nchunk; ++c) {
            const int h = tab[c * E + e];
            tab[c * E + e] = run;
            run += h;
        }
        off_s[e] = run;                  // the count, for now
        run_kept += (int)min((int64_t)run, cap);
    }
    scan_s[threadIdx.x] = run_kept;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {
        const int add = threadIdx.x >= o ? scan_s[threadIdx.x - o] : 0;
        __syncthreads();
        scan_s[threadIdx.x] += add;
        __syncthreads();
    }
    int before = scan_s[threadIdx.x] - run_kept;
    for (int e = e0; e < e1; ++e) {
        const int cnt = off_s[e];
        const int kp = (int)min((int64_t)cnt, cap);
        if (blockIdx.x == 0) {
            counts[e] = cnt;
            kept[e] = kp;
            offsets[e] = before;
        }
        off_s[e] = before;
        before += kp;
    }
    if (threadIdx.x == 255) {
        off_s[E] = scan_s[255];
        if (blockIdx.x == 0) offsets[E] = scan_s[255];
    }
    __syncthreads();
    // unused tail of perm -> -1
    {
        const int64_t used = off_s[E];
        const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        const int64_t gsz = (int64_t)gridDim.x * blockDim.x;
        for (int64_t i = used + gtid; i < S; i += gsz) perm[i] = -1;
    }
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_row = -1;
    if (lane < k) {
        const int64_t sl = t * k + lane;
        const int e = __ldg(idx + sl);
        if (e >= 0 && e < E) {
            const int64_t pr = (int64_t)lane * T + t;           // priority of slot (t, lane)
            const int rank = tab[(pr / lchunk) * E + e] + __ldg(lrank + sl);
            if ((int64_t)rank < cap) {
                my_row = off_s[e] + rank;
                perm[my_row] = (int32_t)sl;
            }
        }
        inv[sl] = my_row;                                        // -1: dropped or invalid (flagged earlier)
    }
    int rows[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(kFull, my_row, j);
    const uint4 *src = x + t * nvec;
    int64_t v = lane;
    for (; v + 96 < nvec; v += 128) {
        uint4 a0 = __ldg(src + v), a1 = __ldg(src + v + 32), a2 = __ldg(src + v + 64),
              a3 = __ldg(src + v + 96);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j < k && rows[j] >= 0) {
                uint4 *dst = x_perm + (int64_t)rows[j] * nvec;
                dst[v] = a0;
                dst[v + 32] = a1;
                dst[v + 64] = a2;
                dst[v + 96] = a3;
            }
        }
    }
    for (; v < nvec; v += 32) {
        const uint4 a = __ldg(src + v);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < k && rows[j] >= 0) x_perm[(int64_t)rows[j] * nvec + v] = a;
    }
}

// Whole integer dispatch in one CTA of 1024 threads, for layers of at most
// kSmallSlots slots and kSmallExperts experts.  The top-k indices are first
// copied into shared memory (16-bit, one vectorised pass), then warp w owns
// priorities [w*span, (w+1)*span): per-warp histograms -> per-expert warp
// bases (an exclusive scan over warps in warp order, which is priority
// order) -> counts, kept, offsets -> match-any ranks -> perm, inv.  Same
// result as the chunked kernels, two launches fewer.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;

__global__ void __launch_bounds__(kSmallThreads) perm_small_kernel(const int32_t *idx, int T, int k, int E,
                                                                   int64_t cap, int32_t *counts, int32_t *kept,
                                                                   int32_t *offsets, int32_t *perm, int32_t *inv,
                                                                   int32_t *err) {
    PDL_ENTER();
    extern __shared__ int wh[];            // [kSmallWarps][E] histograms, then warp bases; then slot experts
    __shared__ int warp_tot[32];
    short *es = reinterpret_cast<short *>(wh + kSmallWarps * E);   // [S] expert of slot s (-2: invalid)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = T * k;
    const int span = ((S + kSmallWarps - 1) / kSmallWarps + 31) / 32 * 32;   // multiple of 32
    for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) wh[i] = 0;
    // expert ids, slot order (t*k + j); 16-byte loads while aligned
    const int nvec = ((S & 3) == 0 && (reinterpret_cast<uintptr_t>(idx) & 15) == 0) ? S / 4 : 0;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int4 q = __ldg(reinterpret_cast<const int4 *>(idx) + v);
        const int a[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) es[4 * v + h] = (short)((a[h] >= 0 && a[h] < E) ? a[h] : -2);
    }
    for (int i = 4 * nvec + threadIdx.x; i < S; i += blockDim.x) {
        const int a = __ldg(idx + i);
        es[i] = (short)((a >= 0 && a < E) ? a : -2);
    }
    __syncthreads();
    const int p0 = warp * span;
    int *my = wh + warp * E;
    // priority p = j*T + t  ->  slot s = t*k + j
    auto slot_of = [&](int p) { const int j = p / T; return (p - j * T) * k + j; };
    for (int g = 0; g < span; g += 32) {
        const int p = p0 + g + lane;
        if (p < S) {
            const int e = es[slot_of(p)];
            if (e >= 0) atomicAdd(&my[e], 1);
            else atomicExch(err, 1);       // MOE_ERR_INVALID_ARG
        }
    }
    __syncthreads();
    int kp_mine = 0;
    if ((int)threadIdx.x < E) {
        const int e = threadIdx.x;
        int run = 0;
        for (int w = 0; w < kSmallWarps; ++w) {
            const int c = wh[w * E + e];
            wh[w * E + e] = run;
            run += c;
        }
        counts[e] = run;
        kp_mine = (int64_t)run < cap ? run : (int)cap;
        kept[e] = kp_mine;
    }
    // exclusive block scan of kept -> offsets (kept in shared memory too)
    int v = kp_mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += u;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + v - kp_mine;
    __shared__ int off_s[kSmallExperts + 1];
    if ((int)threadIdx.x < E) {
        offsets[threadIdx.x] = before;
        off_s[threadIdx.x] = before;
    }
    if ((int)threadIdx.x == E - 1) offsets[E] = before + kp_mine;
    __syncthreads();
    // ranks in priority order, 32 slots at a time
    const unsigned lt = (1u << lane) - 1u;
    for (int g = 0; g < span; g += 32) {
        const int p = p0 + g + lane;
        int s = -1, e = -1;
        if (p < S) {
            s = slot_of(p);
            e = es[s];
        }
        const unsigned peers = __match_any_sync(kFull, e);
        int rank = 0;
        if (e >= 0) rank = my[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && (peers & lt) == 0) my[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            if ((int64_t)rank < cap) {
                const int row = off_s[e] + rank;
                perm[row] = s;
                inv[s] = row;
            } else {
                inv[s] = -1;
            }
        } else if (e == -2) {
            inv[s] = -1;
        }
    }
}

__global__ void __launch_bounds__(256) perm_copy_kernel(const uint4 *x, int64_t T, int k, int64_t nvec,
                                                        const int32_t *inv, const int32_t *offsets,
                                                        int E, int32_t *perm, int64_t S, uint4 *x_perm) {
    PDL_ENTER();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    // unused tail of perm -> -1
    {
        const int64_t used = offsets[E];
        const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        const int64_t gsz = (int64_t)gridDim.x * blockDim.x;
        for (int64_t i = used + gtid; i < S; i += gsz) perm[i] = -1;
    }
    if (t >= T) return;
    int rows[kMaxTopK];
    const int my_row = lane < k ? inv[t * k + lane] : -1;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(kFull, my_row, j);
    const uint4 *src = x + t * nvec;
    int64_t v = lane;
    for (; v + 96 < nvec; v += 128) {
        uint4 a0 = __ldg(src + v), a1 = __ldg(src + v + 32), a2 = __ldg(src + v + 64),
              a3 = __ldg(src + v + 96);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j < k && rows[j] >= 0) {
                uint4 *dst = x_perm + (int64_t)rows[j] * nvec;
                dst[v] = a0;
                dst[v + 32] = a1;
                dst[v + 64] = a2;
                dst[v + 96] = a3;
            }
        }
    }
    for (; v < nvec; v += 32) {
        const uint4 a = __ldg(src + v);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < k && rows[j] >= 0) x_perm[(int64_t)rows[j] * nvec + v] = a;
    }
}

}  // namespace

// Scratch of the allocation-free dispatch entry point: the chunk histogram
// table followed by the chunk base table, kPermStaticScratchInts int32 in
// total (512 KB), resident on every device that loads the library.  Host
// code must not use this name as an address; permute_static_scratch()
// returns the device address.
static __device__ __align__(256) int32_t g_perm_static_scratch[kPermStaticScratchInts];

int32_t *permute_static_scratch() {
    // one cudaGetSymbolAddress per device (and per context of that device),
    // made with that device current
    static SymbolCache cache;
    return static_cast<int32_t *>(symbol_address(cache, (const void *)g_perm_static_scratch));
}

cudaError_t launch_permute(const PermuteParams &p, cudaStream_t s) {
    const int64_t S = p.T * p.k;
    const int64_t nchunk = ceil_div(S, kPermChunk);
    int32_t *err = device_error_flag();
    if (!err) return cudaErrorUnknown;
    const int eb = p.dtype == 0 ? 4 : 2;
    const int64_t nvec = (int64_t)p.d * eb / 16;
    const dim3 copy_grid((unsigned)ceil_div(p.T, 8));
    cudaError_t e;
    if (!p.chunked && S > 0 && S <= kSmallSlots && p.E <= kSmallExperts) {
        const size_t smem = (size_t)kSmallWarps * p.E * sizeof(int) + (size_t)S * sizeof(short);
        if (smem > 48 * 1024) {
            e = cudaFuncSetAttribute(perm_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        e = launch_pdl(perm_small_kernel, dim3(1), dim3(kSmallThreads), smem, s, p.topk_idx, (int)p.T, p.k, p.E,
                       p.cap, p.counts, p.kept, p.offsets, p.perm, p.inv, err);
        if (e != cudaSuccess) return e;
        return launch_pdl(perm_copy_kernel, copy_grid, dim3(256), 0, s, static_cast<const uint4 *>(p.x), p.T, p.k,
                          nvec, p.inv, p.offsets, p.E, p.perm, S, static_cast<uint4 *>(p.x_perm));
    }
    int lchunk = kLocalChunkMin;
    while (lchunk < kPermChunk && ceil_div(S, lchunk) * p.E > kTwoPassTable) lchunk *= 2;
    const int64_t nlocal = ceil_div(S, lchunk);
    if (!p.chunked && nlocal > 0 && nlocal * p.E <= kTwoPassTable) {
        const size_t smem1 = (size_t)(kPermThreads / 32) * p.E * sizeof(int);
        if (smem1 > 48 * 1024) {
            e = cudaFuncSetAttribute(perm_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
            if (e != cudaSuccess) return e;
        }
        e = launch_pdl(perm_local_kernel, dim3((unsigned)nlocal), dim3(kPermThreads), smem1, s, p.topk_idx, p.T,
                       p.k, p.E, lchunk, p.hist, p.lrank, err);
        if (e != cudaSuccess) return e;
        const size_t smem2 = (size_t)(nlocal * p.E + p.E + 1) * sizeof(int);
        if (smem2 > 48 * 1024) {
            e = cudaFuncSetAttribute(perm_copy_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(perm_copy_rank_kernel, copy_grid, dim3(256), smem2, s, static_cast<const uint4 *>(p.x), p.T,
                          p.k, nvec, p.topk_idx, p.E, p.cap, lchunk, nlocal, p.hist, p.lrank, p.counts, p.kept,
                          p.offsets,
                          p.perm, p.inv, static_cast<uint4 *>(p.x_perm));
    }
    if (nchunk > 0) {
        e = launch_pdl(perm_hist_kernel, dim3((unsigned)nchunk), dim3(kPermThreads), p.E * sizeof(int), s,
                       p.topk_idx, p.T, p.k, p.E, p.hist, err);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, p.hist, p.base, nchunk, p.E, p.cap, p.counts,
                   p.kept, p.offsets);
    if (e != cudaSuccess || nchunk == 0) return e;
    const size_t rank_smem = (size_t)(kPermThreads / 32) * p.E * sizeof(int);
    if (rank_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(perm_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rank_smem);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(perm_rank_kernel, dim3((unsigned)nchunk), dim3(kPermThreads), rank_smem, s, p.topk_idx, p.T,
                   p.k, p.E, p.cap, p.base, p.offsets, p.perm, p.inv, err);
    if (e != cudaSuccess) return e;
    return launch_pdl(perm_copy_kernel, copy_grid, dim3(256), 0, s, static_cast<const uint4 *>(p.x), p.T, p.k, nvec,
                      p.inv, p.offsets, p.E, p.perm, S, static_cast<uint4 *>(p.x_perm));
}

}  // namespace moe
