// Grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA loads) for the expert FFNs and the router of wide
// layers.
//
//   out[r, n] = epilogue( sum_k A[r, k] * B[g * b_group_rows + n, k] )
//
// for every row r of group g (rows seg[g] .. seg[g+1]-1 of A).  A is the
// permuted token matrix (experts' segments are contiguous) and B the stacked
// expert weights in nn.Linear layout, so both operands are K-major.  The
// epilogue adds the bias and applies GELU / ReLU, or for a gated (SwiGLU)
// layer multiplies silu(A W1^T) by A W3^T; the two products share one MMA
// (the B tile stacks BN/2 rows of W1 over BN/2 rows of W3, so accumulator
// columns [0, BN/2) are the gate and [BN/2, BN) the up projection).
//
// Pages: "MoE Training: Mixture of Experts" (Quick Start expert Linear-GELU-
// Linear); "moe_code.py" (Expert: ReLU FFN); the Mixtral parameter
// arithmetic of the MoE technical survey (three-matrix SwiGLU expert).
//
// Structure: one persistent CTA per SM, 320 threads.
//   warp 0      TMA producer: A tile 128x64 and B tile BNx64 per stage,
//               128-byte swizzle, completion on an mbarrier (expect_tx).
//   warp 1      TMEM allocator and MMA issuer: 4 x tcgen05.mma
//               (M=128, N=BN, K=16, bf16 -> fp32) per stage, tcgen05.commit
//               frees the stage and, after the last K block, publishes the
//               accumulator.
//   warps 2-9   epilogue, two warps per TMEM lane quadrant (warp w reads
//               lanes 32*(w%4) ..) on alternate 32-column chunks:
//               tcgen05.ld, bias/activation in fp32, staged through shared
//               memory into row-contiguous 64-byte segments (whole sectors);
//               then they release the accumulator.
// Two accumulators (2 x BN TMEM columns) let the epilogue of tile i overlap
// the main loop of tile i+1.  Tiles are ordered group-major, then N-block,
// then M-block, so the CTAs working at the same time share weight tiles.
// Every wait is bounded: a wait that gives up raises the library's device
// error flag and an abort flag in shared memory, every role leaves its
// loop, copies and MMAs in flight are drained (again bounded) and TMEM is
// released before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "moe_internal.h"
#include "route_device.cuh"

namespace moe {

// ------------------------------------------------------------------ device flag
__device__ int32_t g_moe_device_error = 0;

// The context current on this thread (the driver's cuCtxGetCurrent, looked
// up through the runtime so that the library does not link the driver).
static void *current_context() {
    using Fn = CUresult (*)(CUcontext *);
    static Fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<Fn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

void *symbol_address(SymbolCache &cache, const void *symbol) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SymbolCache::kDevices) return nullptr;
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(cache.mu);
    if (!cache.ptr[dev] || !ctx || cache.ctx[dev] != ctx) {
        void *p = nullptr;
        // (makes the device's primary context current if no context was)
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
        cache.ptr[dev] = p;
        cache.ctx[dev] = current_context();
    }
    return cache.ptr[dev];
}

int32_t *device_error_flag() {
    static SymbolCache cache;
    return static_cast<int32_t *>(symbol_address(cache, (const void *)&g_moe_device_error));
}

// Process-wide switches set through moe_set_option (defaults: programmatic
// dependent launch on, GEMM kernel chosen by shape, 2 s device waits).
namespace {
std::atomic<int64_t> g_opt_pdl{1};
std::atomic<int64_t> g_opt_gemm_pair{-1};
std::atomic<int64_t> g_opt_wait_ns{2000000000ll};
std::atomic<int64_t> g_opt_gemm_band{-1};
}  // namespace

bool pdl_enabled() { return g_opt_pdl.load(std::memory_order_relaxed) != 0; }
int gemm_pair_option() { return (int)g_opt_gemm_pair.load(std::memory_order_relaxed); }
uint64_t wait_limit_ns() { return (uint64_t)g_opt_wait_ns.load(std::memory_order_relaxed); }
int64_t gemm_band_option() { return g_opt_gemm_band.load(std::memory_order_relaxed); }

bool set_option(int option, int64_t value) {
    switch (option) {
        case 0:   // MOE_OPT_PDL
            if (value != 0 && value != 1) return false;
            g_opt_pdl.store(value);
            return true;
        case 1:   // MOE_OPT_GEMM_PAIR
            if (value < -1 || value > 1) return false;
            g_opt_gemm_pair.store(value);
            return true;
        case 2:   // MOE_OPT_WAIT_LIMIT_NS
            if (value < 0) return false;
            g_opt_wait_ns.store(value);
            return true;
        case 3:   // MOE_OPT_GEMM_BAND
            if (value < -1 || value > 65536) return false;
            g_opt_gemm_band.store(value);
            return true;
        default:
            return false;
    }
}
bool get_option(int option, int64_t *value) {
    switch (option) {
        case 0: *value = g_opt_pdl.load(); return true;
        case 1: *value = g_opt_gemm_pair.load(); return true;
        case 2: *value = g_opt_wait_ns.load(); return true;
        case 3: *value = g_opt_gemm_band.load(); return true;
        default: return false;
    }
}

int num_sms() {
    static int n[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!n[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        n[dev] = v > 0 ? v : 148;
    }
    return n[dev];
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                 // one 128-byte swizzle atom of bf16
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 8;   // two per TMEM lane quadrant (default); a CTA is 64 + 32 EW threads
// The plain bf16-output kernel of GELU / ReLU layers takes 16 epilogue
// warps (four per quadrant): at d_model 1024 its activation math, not the
// tensor cores, bounds a tile.
constexpr int kEpiWarpsWide = 16;
constexpr uint64_t kDrainLimitNs = 2000000000ull;  // teardown waits: 2 s, whatever the wait limit

template <int BN, int EW = kEpiWarps>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN >= 256 ? 4 : (BN >= 128 ? 6 : (BN >= 64 ? 8 : 10));
    static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr int EPI_BYTES = EW * 32 * 64;   // per epilogue warp: 32 rows x 64 B
    static constexpr int BAR_BYTES = 256;
    static size_t smem_bytes(int G) {
        return 1024 + (size_t)STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + (size_t)2 * (G + 1) * sizeof(int);
    }
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase parity.  Returns false when the CTA is aborting
// (flag already set) or the limit (ns of %globaltimer) ran out (then sets
// both flags).
__device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                            int32_t *err, uint64_t limit_ns) {
    const uint64_t t0 = global_timer();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicExch(err, 6);  // MOE_ERR_DEVICE_TIMEOUT
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag, err, limit_ns);
}
// Wait bounded by time only (teardown: in-flight work must land first, so
// this bound does not follow the configurable wait limit).
__device__ __noinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(bar, parity))
        if (global_timer() - t0 > kDrainLimitNs) return false;
    return true;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, uint64_t *bar, int32_t c0,
                                            int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle,
// 8-row core-matrix groups 1024 bytes apart (SBO), version field 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;              // LBO (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;    // SBO
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// The same for an MN-major operand tile (N contiguous in global memory):
// TMA boxes of 64 K rows x 64 N elements (128 bytes, 128-byte swizzle), one
// per 64-wide N block, 8 KB apart (LBO); 8-row K groups 1 KB apart (SBO).
// One K=16 MMA step advances 16 rows = 2 KB.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(8192 >> 4) << 16;    // LBO: next 64-element N block
    d |= (uint64_t)(1024 >> 4) << 32;    // SBO: next 8-row K group
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, each K-major or
// MN-major (the transpose-A / transpose-B bits).
template <int M, int N, bool B_MN = false, bool A_MN = false>
struct IDesc {
    static constexpr uint32_t value = (1u << 4) | (1u << 7) | (1u << 10) | (A_MN ? (1u << 15) : 0u) |
                                      (B_MN ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
                                      ((uint32_t)(M >> 4) << 24);
};

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 columns of fp32 from TMEM (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ kernel
struct Args {
    const int32_t *seg;
    int64_t a_rows;
    int G, M, N, K, b_group_rows;
    void *out;
    int64_t ldo;
    const bf16 *bias;
    int64_t bias_stride;
    int act;
    int32_t *err;
    RouteEpilogue route;   // router GEMM with the routing epilogue
    bf16 *pre;             // forward: pre-activations written (or null); backward: pre-activations read
    int64_t ld_pre;
    int kgroup;            // 1: groups split K (weight gradients), seg = per-group K offsets
    int64_t out_group_stride;  // K-grouped: elements between the groups' outputs
    int k_split;           // MN-major B: K below k_split from tmB, the rest from tmB2
    int n_inner;           // K-grouped: consecutive tiles walk N (else M) inside a group
    uint64_t wait_ns;      // bound of every mbarrier wait (ns); a wait that runs out aborts the kernel
    // second expert GEMM of the layer forward: rows scaled by their gate,
    // plus x for a token's first kept slot (GemmProblem::comb)
    CombinePrep comb;
    int band;              // M-grouped: M tiles per raster band (0: whole group)
};

struct Tile {
    int g, row0, seg_end, n0;
};

// Tile `tile` of an M-grouped problem: group by binary search over the
// tile prefix, then inside the group bands of `band` M tiles (0: one band
// of the whole group), N block outer and M tile inner within a band, so
// that the tiles in flight share a band's A rows and B columns in L2.
__device__ __forceinline__ Tile decode_tile_m(int tile, const int *seg_s, const int *pre_s, int G, int bn_out,
                                              int tile_m, int band = 0) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre_s[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    const int rows = seg_s[lo + 1] - seg_s[lo];
    const int mt = (rows + tile_m - 1) / tile_m;
    const int local = tile - pre_s[lo];
    int nb, mb;
    if (band <= 0 || band >= mt) {
        nb = local / mt;
        mb = local - nb * mt;
    } else {
        const int nt = (pre_s[lo + 1] - pre_s[lo]) / mt;
        const int per_band = band * nt;
        const int b = local / per_band;
        const int in_rows = min(band, mt - b * band);
        const int in = local - b * per_band;
        nb = in / in_rows;
        mb = b * band + (in - nb * in_rows);
    }
    Tile t;
    t.g = lo;
    t.row0 = seg_s[lo] + mb * tile_m;
    t.seg_end = seg_s[lo + 1];
    t.n0 = nb * bn_out;
    return t;
}
__device__ __forceinline__ Tile decode_tile(int tile, const int *seg_s, const int *pre_s, int G, int bn_out,
                                            int band = 0) {
    return decode_tile_m(tile, seg_s, pre_s, G, bn_out, BM, band);
}

// Gaussian CDF for the GELU epilogues, from the rational approximation of
// erfc in Abramowitz & Stegun, Handbook of Mathematical Functions, 7.1.26
// (after Hastings): for x >= 0, erfc(x) = t (a1 + t (a2 + t (a3 + t (a4 +
// t a5)))) exp(-x^2) + eps, t = 1 / (1 + p x), |eps| <= 1.5e-7.  With
// x = |a| / sqrt(2), Phi(a) = erfc(x) / 2 for a < 0 (no cancellation) and
// 1 - erfc(x) / 2 otherwise; exp(-x^2) = exp(-a^2 / 2) is returned in `e`
// for the density term of GELU'.  One exponential and one reciprocal per
// element, where erff and expf cost the backward epilogue twice as much.
struct ErfcAS7126 {
    static constexpr float p = 0.3275911f, a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                           a4 = -1.453152027f, a5 = 1.061405429f;
};
__device__ __forceinline__ float gauss_cdf(float a, float &e) {
    using K = ErfcAS7126;
    const float x = fabsf(a) * 0.70710678118654752f;
    const float t = __fdividef(1.0f, fmaf(K::p, x, 1.0f));
    e = __expf(-x * x);
    const float half_erfc = 0.5f * t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, K::a5, K::a4), K::a3), K::a2), K::a1) * e;
    return a >= 0.0f ? 1.0f - half_erfc : half_erfc;
}

// Paired fp32 arithmetic (f32x2: two lanes of a 64-bit register per
// instruction), for the activation math of the epilogues.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_splat(float v) { return f2_pack(v, v); }
__device__ __forceinline__ float rcp_approx(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float exp2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// GELU(a) = a Phi(a) of two values: the A&S 7.1.26 evaluation of gauss_cdf
// with the multiplies and the polynomial on paired lanes, Phi(a) from half
// erfc(|a| / sqrt 2) = t (a1 + t (a2 + ...)) exp(-x^2) / 2, where
// exp(-x^2) = 2^(-x^2 log2 e).
__device__ __forceinline__ void gelu_erf2(float &v0, float &v1) {
    using K = ErfcAS7126;
    const uint64_t x = f2_mul(f2_pack(fabsf(v0), fabsf(v1)), f2_splat(0.70710678118654752f));
    float d0, d1;
    f2_unpack(f2_fma(f2_splat(K::p), x, f2_splat(1.0f)), d0, d1);
    const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
    float q0, q1;
    f2_unpack(f2_mul(f2_mul(x, x), f2_splat(-1.4426950408889634f)), q0, q1);   // -x^2 log2 e
    const uint64_t e = f2_pack(exp2_approx(q0), exp2_approx(q1));
    uint64_t poly = f2_fma(t, f2_splat(K::a5), f2_splat(K::a4));
    poly = f2_fma(poly, t, f2_splat(K::a3));
    poly = f2_fma(poly, t, f2_splat(K::a2));
    poly = f2_fma(poly, t, f2_splat(K::a1));
    float h0, h1;
    f2_unpack(f2_mul(f2_mul(t, poly), f2_mul(e, f2_splat(0.5f))), h0, h1);
    const float c0 = v0 >= 0.0f ? 1.0f - h0 : h0, c1 = v1 >= 0.0f ? 1.0f - h1 : h1;
    f2_unpack(f2_mul(f2_pack(v0, v1), f2_pack(c0, c1)), v0, v1);
}
__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

// One 32-column chunk of a warp's 32 rows (thread = row) to global memory,
// staged through the warp's 2 KB shared buffer (16-byte units XOR-swizzled
// by row, conflict-free both ways).  bf16: 32 rows x 64 B in one pass, 8
// rows per warp store.  fp32: the chunk is 128 B per row, so it goes in two
// passes of 16 rows (lanes 0-15, then 16-31) and every warp store writes 4
// whole 128-byte lines.  Rows from row_end and columns from ncols (in
// 16-byte units) are not written.
template <bool OUT_F32>
__device__ __forceinline__ void store_chunk(const float (&v)[32], void *out, int64_t ldo, int col, int ncols,
                                            int row_base, int row_end, uint8_t *stg, int lane) {
    if constexpr (OUT_F32) {
        uint4 *sbuf = reinterpret_cast<uint4 *>(stg);      // [16 rows][8 units]
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
            if ((lane >> 4) == ps) {
                const int r = lane & 15;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    sbuf[r * 8 + (j ^ (r & 7))] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                                             __float_as_uint(v[4 * j + 2]),
                                                             __float_as_uint(v[4 * j + 3]));
            }
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int idx = it * 32 + lane, r = idx >> 3, cc = idx & 7;
                const uint4 val = sbuf[r * 8 + (cc ^ (r & 7))];
                const int grow = row_base + 16 * ps + r;
                if (grow < row_end && col + 4 * cc < ncols)
                    reinterpret_cast<uint4 *>(static_cast<float *>(out) + (int64_t)grow * ldo + col)[cc] = val;
            }
            __syncwarp();
        }
    } else {
        uint4 *srow = reinterpret_cast<uint4 *>(stg + lane * 64);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * j + 2 * h], v[8 * j + 2 * h + 1]);
                w[h] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            srow[j ^ ((lane >> 1) & 3)] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int cidx = it * 32 + lane, r = cidx >> 2, cc = cidx & 3;
            const uint4 val = reinterpret_cast<const uint4 *>(stg + r * 64)[cc ^ ((r >> 1) & 3)];
            if (row_base + r < row_end && col + 8 * cc < ncols)
                reinterpret_cast<uint4 *>(static_cast<bf16 *>(out) + (int64_t)(row_base + r) * ldo + col)[cc] = val;
        }
        __syncwarp();
    }
}

// 32 bf16 of this thread's row (row < row_end) as fp32, else zeros.
__device__ __forceinline__ void load_row32_bf16(const bf16 *base, int64_t ld, int row, int row_end, int col,
                                                float (&v)[32]) {
    if (row < row_end) {
        const uint4 *p = reinterpret_cast<const uint4 *>(base + (int64_t)row * ld + col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = __ldg(p + q);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * q + 2 * h] = __uint_as_float(w[h] << 16);
                v[8 * q + 2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
}

// GELU'(a) = Phi(a) + a phi(a), phi(a) = exp(-a^2 / 2) / sqrt(2 pi)
__device__ __forceinline__ float gelu_erf_grad(float a) {
    float e;
    const float c = gauss_cdf(a, e);
    return fmaf(a * 0.39894228040143268f, e, c);
}

// Tile of either kind of problem: M-grouped (rows of A split into groups,
// decode_tile) or K-grouped (every group a full M x N output over its own
// K range; tiles group-major, then N block, then M block).
__device__ __forceinline__ Tile tile_of(const Args &args, int tile, const int *seg_s, const int *pre_s, int G,
                                        int bn_out, int kg_tiles) {
    if (!args.kgroup) return decode_tile(tile, seg_s, pre_s, G, bn_out, args.band);
    const int mt = (args.M + BM - 1) / BM;
    Tile t;
    t.g = tile / kg_tiles;
    const int local = tile - t.g * kg_tiles;
    int mb, nb;
    if (args.n_inner) {
        const int nt = kg_tiles / mt;
        mb = local / nt;
        nb = local - mb * nt;
    } else {
        nb = local / mt;
        mb = local - nb * mt;
    }
    t.row0 = mb * BM;
    t.seg_end = args.M;
    t.n0 = nb * bn_out;
    return t;
}

// K blocks of a tile: M-grouped, all of K; K-grouped, the group's K range
// (64-aligned offsets, block = column / 64); K-grouped MN-major, the
// group's rows seg[g] .. seg[g+1]-1 in blocks of 64 from seg[g] (the last
// block partial).
struct KRange {
    int kb0, kb1;
};
template <bool KG_MN>
__device__ __forceinline__ KRange k_range(const Args &args, const Tile &tl, const int *seg_s, int num_kb) {
    if (KG_MN) return {0, (seg_s[tl.g + 1] - seg_s[tl.g] + BK - 1) / BK};
    if (args.kgroup) return {seg_s[tl.g] / BK, seg_s[tl.g + 1] / BK};
    return {0, num_kb};
}

// Epilogue modes beyond the forward FFN: the activation backward of the
// first expert GEMM, fused into the GEMM that produces dh = dy W2.
constexpr int kEpiBwdGated = 100;   // SwiGLU: da1 = dh a3 silu'(a1), da3 = dh silu(a1)
constexpr int kEpiBwdAct = 101;     // GELU / ReLU: da = dh act'(a)

// Epilogue of one accumulator tile for one warp: rows row_base .. +31 (the
// warp's TMEM lane quadrant q), every PARTS-th 32-column chunk starting at
// 32 * part (PARTS warps share a quadrant).  `out` is this tile's output base (the group's, for K-grouped
// problems); zero_acc: the tile had no K blocks, so its result is zero.
// Shared by the single-CTA and the CTA-pair kernels.
//   forward:  [bias], [pre-activations stored], activation or SwiGLU gating
//   kEpiBwdGated / kEpiBwdAct: the activation backward from the stored
//             pre-activations (args.pre), dh being the accumulator.
template <int BN, bool GATED, bool OUT_F32, int EPI = 0, int PARTS = 2>
__device__ __forceinline__ void epilogue_tile(const Args &args, const Tile &tl, void *out, int row_base,
                                              uint32_t tbase, int part, int lane, uint8_t *stg, bool zero_acc) {
    constexpr int BN_OUT = GATED ? BN / 2 : BN;
    const int row = row_base + lane;
    // combine preparation (fp32 output of a plain GEMM): this row's gate,
    // and the token whose x it adds when it is the token's first kept slot
    constexpr bool kComb = !GATED && OUT_F32 && EPI == 0;
    bool comb = false;
    float cgate = 1.0f;
    int64_t ctok = -1;
    if constexpr (kComb) {
        const CombinePrep &cp = args.comb;
        if (cp.perm && row < tl.seg_end) {
            comb = true;
            const int32_t sl = __ldg(cp.perm + row);
            const int64_t t = sl / cp.k;
            const int j = sl - (int)(t * cp.k);
            cgate = __ldg(cp.gate + sl);
            bool first = cp.x != nullptr;
            for (int jj = 0; jj < j && first; ++jj) first = __ldg(cp.inv + t * cp.k + jj) < 0;
            if (first) ctok = t;
        }
    }
#pragma unroll 1
    for (int c = 32 * part; c < BN_OUT; c += 32 * PARTS) {
        const int col = tl.n0 + c;
        float v[32];
        if (zero_acc) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        } else {
            tmem_ld32(tbase + c, v);
        }
        if constexpr (EPI == kEpiBwdGated) {
            float a1[32], a3[32];
            load_row32_bf16(args.pre, args.ld_pre, row, tl.seg_end, col, a1);
            load_row32_bf16(args.pre, args.ld_pre, row, tl.seg_end, args.N + col, a3);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float sg = 1.0f / (1.0f + expf(-a1[i]));
                const float dh = v[i];
                v[i] = dh * a3[i] * (sg * (1.0f + a1[i] * (1.0f - sg)));   // da1
                a3[i] = dh * a1[i] * sg;                                    // da3 = dh silu(a1)
            }
            store_chunk<false>(v, out, args.ldo, col, args.N, row_base, tl.seg_end, stg, lane);
            store_chunk<false>(a3, out, args.ldo, args.N + col, 2 * args.N, row_base, tl.seg_end, stg, lane);
            continue;
        } else if constexpr (EPI == kEpiBwdAct) {
            float a[32];
            load_row32_bf16(args.pre, args.ld_pre, row, tl.seg_end, col, a);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                v[i] = args.act == 1 ? v[i] * gelu_erf_grad(a[i]) : (a[i] > 0.0f ? v[i] : 0.0f);
            store_chunk<false>(v, out, args.ldo, col, args.N, row_base, tl.seg_end, stg, lane);
            continue;
        } else {
            if (GATED) {
                float u[32];
                if (zero_acc) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = 0.0f;
                } else {
                    tmem_ld32(tbase + BN / 2 + c, u);
                }
                if (args.pre) {   // training forward: a1 | a3 kept for the backward
                    store_chunk<false>(v, args.pre, args.ld_pre, col, args.N, row_base, tl.seg_end, stg, lane);
                    store_chunk<false>(u, args.pre, args.ld_pre, args.N + col, 2 * args.N, row_base, tl.seg_end,
                                       stg, lane);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = silu(v[i]) * u[i];
            } else {
                if (args.bias && col + 32 <= args.N) {
                    const uint4 *bp =
                        reinterpret_cast<const uint4 *>(args.bias + (int64_t)tl.g * args.bias_stride + col);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const uint4 b = __ldg(bp + qq);
                        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            v[qq * 8 + 2 * h] += __uint_as_float(w[h] << 16);
                            v[qq * 8 + 2 * h + 1] += __uint_as_float(w[h] & 0xffff0000u);
                        }
                    }
                }
                if (args.pre && args.act != 0)   // training forward: the pre-activation a
                    store_chunk<false>(v, args.pre, args.ld_pre, col, args.N, row_base, tl.seg_end, stg, lane);
                if (args.act == 1) {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) gelu_erf2(v[i], v[i + 1]);
                } else if (args.act == 2) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.0f);
                }
            }
            if constexpr (kComb) {
                if (comb) {
                    if (ctok >= 0) {
                        float xv[32];
                        load_row32_bf16(args.comb.x, args.N, (int)ctok, (int)ctok + 1, col, xv);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = fmaf(cgate, v[i], xv[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= cgate;
                    }
                }
            }
            store_chunk<OUT_F32>(v, out, args.ldo, col, args.N, row_base, tl.seg_end, stg, lane);
        }
    }
}

// Routing epilogue of the router GEMM (N = E <= EP <= 32, one 32-column
// chunk): thread = token.  The logits (+ router bias) are written, the
// token is routed in registers (route_row), and each warp, whose 32 rows are
// one 32-token block, writes that block's partials: the per-expert sums of
// the softmax probabilities and the expert counts (xor butterflies and
// ballots; lane e keeps expert e) and the sum of lse^2.
template <int EP>
__device__ __forceinline__ void route_epilogue(const Args &args, const Tile &tl, int row_base, const float (&v)[32],
                                               int lane) {
    const RouteEpilogue &re = args.route;
    const int E = args.N;
    const int64_t t = row_base + lane;
    const bool valid = t < tl.seg_end;
    float l[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) l[e] = (e < E && re.b_router) ? v[e] + __ldg(re.b_router + e) : v[e];
    if (valid) {
        float *dst = static_cast<float *>(args.out) + t * args.ldo;
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (e < E) dst[e] = l[e];
    }
    float lse;
    const uint32_t chosen = route_row<EP>(l, E, re.k, re.score_fn, re.renormalize, re.sel_bias, valid, t,
                                          re.topk_idx, re.topk_w, re.lse, &lse);
    if (row_base >= tl.seg_end) return;                  // warp-uniform: no token of this block exists
    const int64_t blk = row_base / 32;
    float ps = 0.0f;
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
        float x = (valid && e < E) ? expf(l[e] - lse) : 0.0f;   // softmax probability
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        const int c = __popc(__ballot_sync(0xffffffffu, (chosen >> e) & 1u));
        if (lane == e) {
            ps = x;
            cnt = c;
        }
    }
    float z = valid ? lse * lse : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < E) {
        re.part_prob[(int64_t)lane * re.nblk + blk] = ps;
        re.part_cnt[(int64_t)lane * re.nblk + blk] = cnt;
    }
    if (lane == 0 && re.part_z) re.part_z[blk] = z;
}

// EPI: 0 forward FFN epilogue; 8 / 16 / 32 routing epilogue (router GEMM,
// E <= EPI); kEpiBwdGated / kEpiBwdAct activation backward.
// KG_MN: K-grouped with both operands MN-major, read in place from the
// row-major token tensors (A [rows, M], B [rows, N]); the group's rows are
// its K range in blocks of 64 from seg[g], and a fixer warp zeroes the K
// rows of a group's last block that belong to the next group.
template <int BN, bool GATED, bool OUT_F32, int EPI = 0, bool B_MN = false, bool KG_MN = false, int EW = kEpiWarps>
__global__ void __launch_bounds__(64 + 32 * EW + (KG_MN ? 32 : 0), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmB2, const Args args) {
    using C = Cfg<BN, EW>;
    constexpr int STAGES = C::STAGES;
    constexpr int BN_OUT = GATED ? BN / 2 : BN;
    constexpr uint32_t IDESC = IDesc<BM, BN, B_MN || KG_MN, KG_MN>::value;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * C::A_BYTES;
    uint8_t *sEpi = smem + STAGES * C::STAGE_BYTES;      // [epilogue warps][32 rows][64 B] staging
    uint64_t *bars = reinterpret_cast<uint64_t *>(sEpi + C::EPI_BYTES);
    uint64_t *full = bars;                 // [STAGES]
    uint64_t *empty = bars + STAGES;       // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;   // [2]
    uint64_t *tempty = tfull + 2;          // [2]
    uint64_t *drain = tempty + 2;          // [1]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *consumed = abort_flag + 1;
    // KG_MN: [STAGES] stage ready for the MMA, after drain and the flags
    uint64_t *fixed = bars + 2 * STAGES + 8;
    static_assert(!KG_MN || (3 * STAGES + 8) * 8 <= C::BAR_BYTES, "barrier area too small");
    int *seg_s = reinterpret_cast<int *>(smem + STAGES * C::STAGE_BYTES + C::EPI_BYTES + C::BAR_BYTES);
    int *pre_s = seg_s + (args.G + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = args.G;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            // KG_MN: a stage is free once the MMAs are done and the fixer has seen it
            mbar_init(&empty[i], KG_MN ? 2 : 1);
            if (KG_MN) mbar_init(&fixed[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 32 * EW);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (GATED) tma_prefetch_desc(&tmB2);
    }
    if (warp == 1) tmem_alloc(tmem_holder, C::TMEM_COLS);
    PDL_ENTER();   // the segment offsets and A are the previous kernel's output
    for (int i = threadIdx.x; i <= G; i += blockDim.x)
        seg_s[i] = args.seg ? args.seg[i] : (i == 0 ? 0 : args.M);
    __syncthreads();
    // tile prefix over groups: n_tiles * ceil(rows_g / BM); K-grouped: every
    // group has ceil(M / BM) * n_tiles tiles, and its K offsets must be
    // multiples of BK (whole, 16-byte aligned TMA boxes) inside K
    const int n_tiles = (args.N + BN_OUT - 1) / BN_OUT;
    const int kg_tiles = ((args.M + BM - 1) / BM) * n_tiles;
    volatile int *seg_bad = consumed + 1;
    if (warp == 0) {
        int carry = 0;
        bool bad = seg_s[0] < 0 || (int64_t)seg_s[G] > (args.kgroup ? (int64_t)args.K : args.a_rows);
        for (int b = 0; b < G; b += 32) {
            const int g = b + lane;
            int v = 0;
            if (g < G) {
                const int rows = seg_s[g + 1] - seg_s[g];
                bad |= rows < 0;
                if (args.kgroup) {
                    if (!KG_MN) bad |= (seg_s[g] % BK) != 0 || (seg_s[g + 1] % BK) != 0;
                    v = kg_tiles;
                } else {
                    v = rows > 0 ? ((rows + BM - 1) / BM) * n_tiles : 0;
                }
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (g < G) pre_s[g + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            pre_s[0] = 0;
            *seg_bad = bad ? 1 : 0;
            if (bad) atomicExch(args.err, 1);  // MOE_ERR_INVALID_ARG
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // segments must be monotone and inside A; otherwise the kernel does nothing
    const int total = *seg_bad ? 0 : pre_s[G];
    const int num_kb = (args.K + BK - 1) / BK;
    int issued = 0;  // producer: TMA stages issued

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t ph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile tl = tile_of(args, tile, seg_s, pre_s, G, BN_OUT, kg_tiles);
            const int brow = args.kgroup ? tl.n0 : tl.g * args.b_group_rows + tl.n0;
            const KRange kr = k_range<KG_MN>(args, tl, seg_s, num_kb);
            bool ok = true;
            for (int kb = kr.kb0; kb < kr.kb1; ++kb) {
                if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, args.err, args.wait_ns)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&full[stage], C::STAGE_BYTES);
                if (KG_MN) {
                    // token rows seg[g] + 64 kb .. as K: 64 x 64 boxes along M and N
                    const int y = seg_s[tl.g] + kb * BK;
#pragma unroll
                    for (int j = 0; j < BM / 64; ++j)
                        tma_load_2d(sA + stage * C::A_BYTES + j * 8192, &tmA, &full[stage], tl.row0 + 64 * j, y);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sB + stage * C::B_BYTES + j * 8192, &tmB, &full[stage], tl.n0 + 64 * j, y);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                    continue;
                }
                // the router GEMM (one tile per CTA, all of them streaming at
                // once) starts every tile at its own K block and wraps around,
                // so that concurrent tiles read different column ranges of
                // their rows instead of the same one
                const int kbl = (EPI > 0 && EPI <= 32)
                                    ? kr.kb0 + (kb - kr.kb0 + tile * 13) % (kr.kb1 - kr.kb0)
                                    : kb;
                tma_load_2d(sA + stage * C::A_BYTES, &tmA, &full[stage], kbl * BK, tl.row0);
                if (B_MN) {
                    // B[n][k] = W[g rows + k][n]: 64 x 64 boxes along N
                    const bool lo = kb * BK < args.k_split;
                    const int y = tl.g * args.b_group_rows + (lo ? kb * BK : kb * BK - args.k_split);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sB + stage * C::B_BYTES + j * 8192, lo ? &tmB : &tmB2, &full[stage],
                                    tl.n0 + 64 * j, y);
                } else if (GATED) {
                    tma_load_2d(sB + stage * C::B_BYTES, &tmB, &full[stage], kb * BK, brow);
                    tma_load_2d(sB + stage * C::B_BYTES + (BN / 2) * BK * 2, &tmB2, &full[stage], kb * BK, brow);
                } else {
                    tma_load_2d(sB + stage * C::B_BYTES, &tmB, &full[stage], kbl * BK, brow);
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t ph = 0, fph = 0;
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, args.err, args.wait_ns)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            const Tile tl = tile_of(args, tile, seg_s, pre_s, G, BN_OUT, kg_tiles);
            const KRange kr = k_range<KG_MN>(args, tl, seg_s, num_kb);
            const int kb0 = kr.kb0, kb1 = kr.kb1;
            // KG_MN: a group's partial last block waits for the fixer, the rest for TMA
            const int kg_rows = KG_MN ? seg_s[tl.g + 1] - seg_s[tl.g] : 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                // fixed[] completes only on tail blocks: its parity is tracked per stage
                const bool tail = KG_MN && kg_rows - kb * BK < BK;
                const uint32_t par = tail ? (fph >> stage) & 1u : ph;
                if (tail) fph ^= 1u << stage;
                if (!mbar_wait(tail ? &fixed[stage] : &full[stage], par, abort_flag, args.err, args.wait_ns)) {
                    ok = false;
                    break;
                }
                *consumed = *consumed + 1;
                tc_fence_after();
                const uint64_t adesc = KG_MN ? sdesc_sw128_mn(smem_u32(sA + stage * C::A_BYTES))
                                             : sdesc_sw128(smem_u32(sA + stage * C::A_BYTES));
                const uint64_t bdesc = (B_MN || KG_MN) ? sdesc_sw128_mn(smem_u32(sB + stage * C::B_BYTES))
                                                       : sdesc_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    // K-major: +32 bytes per K step inside the swizzle atom;
                    // MN-major: +16 rows of 128 bytes (encoded >> 4)
                    umma_bf16(d_tmem, adesc + (uint64_t)(kk * (KG_MN ? 128 : 2)),
                              bdesc + (uint64_t)(kk * ((B_MN || KG_MN) ? 128 : 2)), IDESC,
                              (kb > kb0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(&tfull[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
    } else if (KG_MN && warp == 2 + EW) {
        // ------------------------------------------------ K-tail fixer
        // A group's last K block may reach into the next group's rows: those
        // K rows of A are zeroed (whole 128-byte lines of each 64-column box;
        // a zero row of A zeroes the row's products), and of B too where the
        // block runs past the last group's rows (unwritten memory), before
        // the MMA reads the stage; the proxy fence makes the zeros visible to
        // the tensor cores.  Full blocks go to the MMA straight from TMA; the
        // fixer still observes every stage and frees it together with the
        // MMA (empty counts both), so it never falls a ring cycle behind.
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const Tile tl = tile_of(args, tile, seg_s, pre_s, G, BN_OUT, kg_tiles);
            const int rows = seg_s[tl.g + 1] - seg_s[tl.g];
            const KRange kr = k_range<KG_MN>(args, tl, seg_s, num_kb);
            for (int kb = kr.kb0; kb < kr.kb1; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], ph, abort_flag, args.err, args.wait_ns))) {
                    ok = false;
                    break;
                }
                const int valid = rows - kb * BK;
                if (valid < BK) {
                    const int bad_rows = BK - valid;
                    const bool past_end = seg_s[tl.g] + kb * BK + BK > seg_s[G];
                    const int boxes = BM / 64 + (past_end ? BN / 64 : 0);
                    const int lines = bad_rows * boxes;
                    for (int i = lane; i < lines * 8; i += 32) {
                        const int line = i >> 3, chunk = i & 7;
                        const int box = line / bad_rows, r = valid + line % bad_rows;
                        uint8_t *base = box < BM / 64 ? sA + stage * C::A_BYTES + box * 8192
                                                      : sB + stage * C::B_BYTES + (box - BM / 64) * 8192;
                        *reinterpret_cast<uint4 *>(base + r * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&fixed[stage]);
                }
                if (lane == 0) mbar_arrive(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp >= 2 && warp < 2 + EW) {
        // ------------------------------------------------ epilogue
        // Thread = accumulator row.  Warps w, w+4, ... share a TMEM lane
        // quadrant and take every (EW/4)-th 32-column chunk.  Output leaves
        // through a per-warp 2 KB shared-memory buffer (store_chunk):
        // row-contiguous 64-byte segments of bf16, whole 128-byte lines of fp32.
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;       // which chunks: half, half + EW/4, ...
        uint8_t *stg = sEpi + (warp - 2) * (32 * 64);
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile tl = tile_of(args, tile, seg_s, pre_s, G, BN_OUT, kg_tiles);
            // tcgen05.ld below is warp-collective: leave only as a whole warp
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, abort_flag, args.err, args.wait_ns))) break;
            tc_fence_after();
            const int row_base = tl.row0 + q * 32;          // first row of this warp's 32
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if constexpr (EPI > 0 && EPI <= 32) {
                if (half == 0) {
                    float v[32];
                    tmem_ld32(tbase, v);
                    route_epilogue<EPI>(args, tl, row_base, v, lane);
                }
            } else {
                void *out = args.out;
                bool zero_acc = false;
                if (args.kgroup) {
                    out = static_cast<uint8_t *>(args.out) +
                          tl.g * args.out_group_stride * (int64_t)(OUT_F32 ? 4 : 2);
                    zero_acc = seg_s[tl.g + 1] == seg_s[tl.g];
                }
                epilogue_tile<BN, GATED, OUT_F32, EPI, EW / 4>(args, tl, out, row_base, tbase, half, lane, stg,
                                                                 zero_acc);
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
    }
    // ---------------------------------------------------- teardown
    __syncthreads();  // every role has left its loop
    if (warp == 0 && lane == 0 && *abort_flag) {
        // copies issued but never consumed must land before the CTA exits
        for (int i = *consumed; i < issued; ++i)
            if (!mbar_wait_drain(&full[i % STAGES], (uint32_t)((i / STAGES) & 1))) break;
    }
    if (warp == 1 && lane == 0) {
        // every MMA issued by this CTA has completed once the drain barrier flips
        umma_commit(drain);
        mbar_wait_drain(drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
// The same grouped GEMM with tcgen05.mma.cta_group::2 on a cluster of two
// CTAs (the two SMs of a TPC): the pair computes a 256-row x BN tile, each
// CTA holding 128 rows of A and BN/2 rows of B in its shared memory, and
// each CTA's TMEM holding the accumulator of its own 128 rows.  Per SM the
// tensor work per stage is unchanged while the loaded bytes drop from 48 KB
// to 32 KB, so 6 stages fit instead of 4, and A is re-read half as often.
// The even CTA (rank 0) issues the MMAs; both CTAs' TMA loads complete on
// the even CTA's full barriers; commits are multicast to both CTAs.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *tm, uint32_t mbar_cluster, int32_t c0,
                                                 int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(mbar_cluster), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on the mbarrier at this shared offset in both CTAs of the pair
__device__ __forceinline__ void umma_commit_pair_both(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)0x3)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait with cluster-scope acquire (arrivals may come from the peer CTA)
__device__ __noinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               int32_t *err, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((++n & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicExch(err, 6);  // MOE_ERR_DEVICE_TIMEOUT
                return false;
            }
        }
    }
}

template <int BN, int EW = kEpiWarps>
struct PairCfg {
    static constexpr int A_BYTES = BM * BK * 2;              // 128 rows of A
    static constexpr int B_BYTES = (BN / 2) * BK * 2;        // BN/2 rows of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // per CTA
    static constexpr int STAGES = 6;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_BYTES = EW * 32 * 64;
    static constexpr int BAR_BYTES = 256;
    static constexpr int THREADS = 64 + 32 * EW;
    static size_t smem_bytes(int G) {
        return 1024 + (size_t)STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + (size_t)2 * (G + 1) * sizeof(int);
    }
};

template <int BN, bool GATED, bool OUT_F32, int EW = kEpiWarps>
__global__ void __launch_bounds__(64 + 32 * EW, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmB2, const Args args) {
    using C = PairCfg<BN, EW>;
    constexpr int STAGES = C::STAGES;
    constexpr int BN_OUT = GATED ? BN / 2 : BN;
    constexpr int TILE_M = 2 * BM;
    constexpr uint32_t IDESC = IDesc<TILE_M, BN>::value;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * C::A_BYTES;
    uint8_t *sEpi = smem + STAGES * C::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sEpi + C::EPI_BYTES);
    uint64_t *full = bars;                 // [STAGES] used in the even CTA
    uint64_t *empty = bars + STAGES;       // [STAGES] both CTAs
    uint64_t *tfull = bars + 2 * STAGES;   // [2] both CTAs
    uint64_t *tempty = tfull + 2;          // [2] used in the even CTA
    uint64_t *drain = tempty + 2;          // [1]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *seg_bad = abort_flag + 1;
    int *seg_s = reinterpret_cast<int *>(smem + STAGES * C::STAGE_BYTES + C::EPI_BYTES + C::BAR_BYTES);
    int *pre_s = seg_s + (args.G + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = args.G;
    const uint32_t rank = cluster_rank();
    const int cid = (int)cluster_index(), ncl = (int)cluster_count();

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 2 * EW);   // one arrival per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (GATED) tma_prefetch_desc(&tmB2);
    }
    if (warp == 1) tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
    PDL_ENTER();   // the segment offsets and A are the previous kernel's output
    for (int i = threadIdx.x; i <= G; i += C::THREADS)
        seg_s[i] = args.seg ? args.seg[i] : (i == 0 ? 0 : args.M);
    __syncthreads();
    const int n_tiles = (args.N + BN_OUT - 1) / BN_OUT;
    if (warp == 0) {
        int carry = 0;
        bool bad = seg_s[0] < 0 || (int64_t)seg_s[G] > args.a_rows;
        for (int b = 0; b < G; b += 32) {
            const int g = b + lane;
            int v = 0;
            if (g < G) {
                const int rows = seg_s[g + 1] - seg_s[g];
                bad |= rows < 0;
                v = rows > 0 ? ((rows + TILE_M - 1) / TILE_M) * n_tiles : 0;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (g < G) pre_s[g + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            pre_s[0] = 0;
            *seg_bad = bad ? 1 : 0;
            if (bad && rank == 0) atomicExch(args.err, 1);  // MOE_ERR_INVALID_ARG
        }
    }
    tc_fence_before();
    cluster_sync_all();      // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int total = *seg_bad ? 0 : pre_s[G];
    const int num_kb = (args.K + BK - 1) / BK;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        int stage = 0;
        uint32_t ph = 0;
        for (int tile = cid; tile < total; tile += ncl) {
            const Tile tl = decode_tile_m(tile, seg_s, pre_s, G, BN_OUT, TILE_M, args.band);
            const int arow = tl.row0 + BM * (int)rank;
            const int brow = GATED ? tl.g * args.b_group_rows + tl.n0
                                   : tl.g * args.b_group_rows + tl.n0 + (BN / 2) * (int)rank;
            const CUtensorMap *bmap = (GATED && rank == 1) ? &tmB2 : &tmB;
            bool ok = true;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait_cluster(&empty[stage], ph ^ 1u, abort_flag, args.err, args.wait_ns)) {
                    ok = false;
                    break;
                }
                if (rank == 0) mbar_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                const uint32_t leader_full = map_to_rank(&full[stage], 0);
                tma_load_2d_pair(sA + stage * C::A_BYTES, &tmA, leader_full, kb * BK, arow);
                tma_load_2d_pair(sB + stage * C::B_BYTES, bmap, leader_full, kb * BK, brow);
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ MMA issuer (even CTA)
        int stage = 0;
        uint32_t ph = 0;
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
            if (!mbar_wait_cluster(&tempty[acc], aph ^ 1u, abort_flag, args.err, args.wait_ns)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait_cluster(&full[stage], ph, abort_flag, args.err, args.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = sdesc_sw128(smem_u32(sA + stage * C::A_BYTES));
                const uint64_t bdesc = sdesc_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    umma_bf16_pair(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), IDESC,
                                   (kb > 0 || kk > 0) ? 1u : 0u);
                umma_commit_pair_both(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_pair_both(&tfull[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        uint8_t *stg = sEpi + (warp - 2) * (32 * 64);
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = cid; tile < total; tile += ncl) {
            const Tile tl = decode_tile_m(tile, seg_s, pre_s, G, BN_OUT, TILE_M, args.band);
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(&tfull[acc], aph, abort_flag, args.err, args.wait_ns))) break;
            tc_fence_after();
            const int row_base = tl.row0 + BM * (int)rank + q * 32;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            epilogue_tile<BN, GATED, OUT_F32, 0, EW / 4>(args, tl, args.out, row_base, tbase, half, lane, stg, false);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(&tempty[acc], 0));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
    }
    // ---------------------------------------------------- teardown
    __syncthreads();
    if (warp == 1 && lane == 0 && rank == 0) {
        // every MMA of the pair has completed once the drain barrier flips
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(drain))
                     : "memory");
        mbar_wait_drain(drain, 0);
    }
    if (warp == 0 && lane == 0 && *abort_flag) {
        // the copies of an aborted CTA complete on the even CTA's barriers;
        // give any still in flight time to land before the CTA exits
        const uint64_t t0 = global_timer();
        while (global_timer() - t0 < 1000000ull) {
        }
    }
    tc_fence_before();
    cluster_sync_all();      // neither CTA leaves while the pair still uses its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows, inner] (row-major), box [box_rows, 64], 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows,
               uint64_t ld = 0) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {(ld ? ld : inner) * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Raster band of an M-grouped problem: W tiles run at once, each reading an
// A strip (tile_m rows) and a B strip (b_rows rows) over the whole K.
// While a group's A rows fit in a third of L2 (42 MB), M-fastest over the
// whole group reads every operand once (measured, Mixtral first GEMM: 2.2
// GB read with whole groups, 4.0 GB with bands).  Above that, a band of m
// M tiles puts m A strips and W/m B strips in flight, least bytes at
// m = sqrt(W * b_rows / tile_m) (Mixtral second GEMM: 4.6 GB read instead
// of 5.2).  The MOE_OPT_GEMM_BAND option overrides the choice.
int raster_band(const GemmProblem &p, int W, int tile_m, int b_rows) {
    const int64_t opt = gemm_band_option();
    if (opt >= 0) return (int)opt;
    const int groups = p.seg ? p.G : 1;
    const int64_t group_a_bytes = p.a_rows / std::max(1, groups) * (int64_t)p.K * 2;
    if (group_a_bytes <= (int64_t)42 << 20) return 0;
    return std::max(1, (int)lround(std::sqrt((double)W * b_rows / tile_m)));
}

template <int BN, bool GATED, bool OUT_F32, int EPI = 0, bool B_MN = false, bool KG_MN = false, int EW = kEpiWarps>
cudaError_t launch_t(const GemmProblem &p, cudaStream_t s) {
    using C = Cfg<BN, EW>;
    constexpr int BN_B = GATED ? BN / 2 : BN;   // rows per TMA box of B
    CUtensorMap ta, tb, tb2;
    if (KG_MN) {
        // A [K rows, M cols] and B [K rows, N cols], row strides lda / ldb
        if (!make_tmap(&ta, p.A, (uint64_t)p.M, (uint64_t)p.K, 64, (uint64_t)p.lda)) return cudaErrorInvalidValue;
        if (!make_tmap(&tb, p.B, (uint64_t)p.N, (uint64_t)p.K, 64, (uint64_t)p.ldb)) return cudaErrorInvalidValue;
        tb2 = tb;
    } else if (!make_tmap(&ta, p.A, (uint64_t)p.K, (uint64_t)p.a_rows, BM)) {
        return cudaErrorInvalidValue;
    }
    if (B_MN && !KG_MN) {
        // B stored [groups * K rows][N cols] (N contiguous): 64 x 64 boxes
        if (!make_tmap(&tb, p.B, (uint64_t)p.N, (uint64_t)p.b_rows_total, 64)) return cudaErrorInvalidValue;
        if (p.B2) {
            if (!make_tmap(&tb2, p.B2, (uint64_t)p.N, (uint64_t)p.b_rows_total, 64)) return cudaErrorInvalidValue;
        } else {
            tb2 = tb;
        }
    } else if (!KG_MN && !make_tmap(&tb, p.B, (uint64_t)p.K, (uint64_t)p.b_rows_total, BN_B)) {
        return cudaErrorInvalidValue;
    }
    if (GATED) {
        if (!make_tmap(&tb2, p.B2, (uint64_t)p.K, (uint64_t)p.b_rows_total, BN_B)) return cudaErrorInvalidValue;
    } else if (!B_MN && !KG_MN) {
        tb2 = tb;
    }
    Args a{};
    a.seg = p.seg;
    a.a_rows = p.a_rows;
    a.G = p.seg ? p.G : 1;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.b_group_rows = p.b_group_rows;
    a.out = p.out;
    a.ldo = p.ldo;
    a.bias = p.bias;
    a.bias_stride = p.bias_stride;
    a.act = p.act;
    a.err = device_error_flag();
    if (!a.err) return cudaErrorUnknown;
    a.wait_ns = wait_limit_ns();
    a.comb = p.comb;
    a.band = (p.kgroup || p.route) ? 0 : raster_band(p, num_sms(), BM, BN);
    a.route = p.route ? *p.route : RouteEpilogue{};
    a.pre = p.pre;
    a.ld_pre = p.ld_pre;
    a.kgroup = p.kgroup;
    a.out_group_stride = p.out_group_stride;
    a.k_split = p.B2 ? p.k_split : p.K;
    // K-grouped: of the two tile orders inside a group, the one whose wave of
    // concurrent tiles (one per SM) touches fewer operand rows (A tiles x BM
    // + B tiles x BN), so that a wave's operands stay in L2
    a.n_inner = 0;
    if (p.kgroup) {
        const int64_t W = num_sms();
        const int64_t mt = ((int64_t)p.M + BM - 1) / BM, nt = ((int64_t)p.N + BN_B - 1) / BN_B;
        const int64_t fm = std::min(mt, W) * BM + std::min(nt, (W + mt - 1) / mt) * BN;
        const int64_t fn = std::min(nt, W) * BN + std::min(mt, (W + nt - 1) / nt) * BM;
        a.n_inner = fn < fm ? 1 : 0;
    }
    // MN-major B: the whole 227 KB are reserved, so that every shared-memory
    // address the tensor cores derive from the descriptors lies inside the
    // CTA's allocation
    const size_t smem = (B_MN || KG_MN) ? (size_t)232448 : C::smem_bytes(a.G);
    if ((B_MN || KG_MN) && C::smem_bytes(a.G) > smem) return cudaErrorInvalidValue;
    auto kern = grouped_gemm_kernel<BN, GATED, OUT_F32, EPI, B_MN, KG_MN, EW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(num_sms()), dim3(64 + 32 * EW + (KG_MN ? 32 : 0)), smem, s, ta, tb, tb2, a);
}

template <int BN, bool GATED, bool OUT_F32, int EW = kEpiWarps>
cudaError_t launch_pair_t(const GemmProblem &p, cudaStream_t s) {
    using C = PairCfg<BN, EW>;
    constexpr int BOX_B = BN / 2;   // rows of B per CTA
    CUtensorMap ta, tb, tb2;
    if (!make_tmap(&ta, p.A, (uint64_t)p.K, (uint64_t)p.a_rows, BM)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, p.B, (uint64_t)p.K, (uint64_t)p.b_rows_total, BOX_B)) return cudaErrorInvalidValue;
    if (GATED) {
        if (!make_tmap(&tb2, p.B2, (uint64_t)p.K, (uint64_t)p.b_rows_total, BOX_B)) return cudaErrorInvalidValue;
    } else {
        tb2 = tb;
    }
    Args a{};
    a.seg = p.seg;
    a.a_rows = p.a_rows;
    a.G = p.seg ? p.G : 1;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.b_group_rows = p.b_group_rows;
    a.out = p.out;
    a.ldo = p.ldo;
    a.bias = p.bias;
    a.bias_stride = p.bias_stride;
    a.act = p.act;
    a.err = device_error_flag();
    if (!a.err) return cudaErrorUnknown;
    a.wait_ns = wait_limit_ns();
    a.comb = p.comb;
    // (bands measured no better for CTA pairs: Mixtral second GEMM 6.7 GB
    // read with bands of 9 pair tiles, 6.4 GB M-fastest)
    a.band = gemm_band_option() > 0 ? (int)gemm_band_option() : 0;
    const size_t smem = C::smem_bytes(a.G);
    auto kern = grouped_gemm_pair_kernel<BN, GATED, OUT_F32, EW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms() / 2 * 2), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// CTA pairs pay off when groups are tall (a pair tile covers 256 rows, so
// short expert segments would waste most of it).  Measured on B300: they
// lose for the gated first expert GEMM (Mixtral shape: 6.29 vs 5.97 ms);
// for the second (no activation) they win (Quick Start shape, K = 4096:
// 0.112 vs 0.125 ms; Mixtral shape, K = 14336: 3.12 vs 3.23 and 3.17 vs
// 3.22 ms in two runs), so they run the second GEMM of tall groups.  For
// the GELU / ReLU first GEMM (Quick Start shape) pairs with 8 or 16
// epilogue warps measured no faster than one CTA with 16 (0.125-0.128 ms
// each).  The MOE_OPT_GEMM_PAIR option forces the choice (the tests run both kernels
// on the same shapes).
bool use_pair(const GemmProblem &p) {
    const int opt = gemm_pair_option();
    if (opt == 0 || opt == 1) return opt == 1;
    const int groups = p.seg ? p.G : 1;
    const int64_t rows_per_group = p.a_rows / (groups > 0 ? groups : 1);
    return rows_per_group >= 1024 && p.act == 0 && !p.gated && !p.route;
}

}  // namespace

// Columns are written in 16-byte units: N % 4 == 0 for fp32 output, N % 8
// for bf16; a bias needs whole 32-column chunks.  K % 8 == 0 keeps the TMA
// row stride a multiple of 16 bytes.
bool grouped_gemm_supported(int N, int K, int gated, int out_f32, int has_bias) {
    if (N <= 0 || K <= 0 || K % 8 != 0) return false;
    if (N % (out_f32 ? 4 : 8) != 0) return false;
    if ((gated || has_bias) && N % 32 != 0) return false;
    return true;
}

cudaError_t launch_grouped_gemm(const GemmProblem &p, cudaStream_t s) {
    // K-grouped MN-major: K is the rows (the outer TMA dimension), any count
    const bool ok = p.kgroup && p.kg_mn ? (p.out_f32 && p.N % 4 == 0 && p.K >= 0)
                                        : grouped_gemm_supported(p.N, p.K, p.gated, p.out_f32, p.bias != nullptr);
    if (!ok) return cudaErrorInvalidValue;
    if (p.epi_bwd) {
        // dh = dy W2 with the activation backward in the epilogue (bf16 da out)
        if (p.out_f32 || p.gated || p.kgroup || !p.pre || p.bias) return cudaErrorInvalidValue;
        if (p.b_mn)
            return p.epi_bwd == 1 ? launch_t<256, false, false, kEpiBwdGated, true>(p, s)
                                  : launch_t<256, false, false, kEpiBwdAct, true>(p, s);
        return p.epi_bwd == 1 ? launch_t<256, false, false, kEpiBwdGated>(p, s)
                              : launch_t<256, false, false, kEpiBwdAct>(p, s);
    }
    if (p.b_mn) {
        // data gradient with the weights read in place (fp32 out)
        if (p.gated || !p.out_f32 || p.kgroup || p.bias || p.K % 64 || p.N % 64) return cudaErrorInvalidValue;
        return launch_t<256, false, true, 0, true>(p, s);
    }
    if (p.kgroup) {
        // weight gradients: fp32 out, one full M x N output per group
        if (p.gated || !p.out_f32 || p.bias || !p.seg) return cudaErrorInvalidValue;
        if (p.kg_mn) {
            if (p.M % 64 || p.N % 64 || p.lda % 8 || p.ldb % 8) return cudaErrorInvalidValue;
            return launch_t<256, false, true, 0, false, true>(p, s);
        }
        return launch_t<256, false, true>(p, s);
    }
    if (p.route) {
        if (p.N > 32 || p.gated || !p.out_f32 || p.seg || p.bias) return cudaErrorInvalidValue;
        if (p.N <= 8) return launch_t<32, false, true, 8>(p, s);
        if (p.N <= 16) return launch_t<32, false, true, 16>(p, s);
        return launch_t<32, false, true, 32>(p, s);
    }
    if (p.gated) {
        if (use_pair(p)) return p.out_f32 ? launch_pair_t<256, true, true>(p, s) : launch_pair_t<256, true, false>(p, s);
        return p.out_f32 ? launch_t<256, true, true>(p, s) : launch_t<256, true, false>(p, s);
    }
    if (p.out_f32) {
        // narrowest N tile that covers N, unless that leaves most SMs idle:
        // then the N tile shrinks (down to 64) to make more tiles
        const int64_t m_tiles = p.seg ? (p.a_rows + BM - 1) / BM : ((int64_t)p.M + BM - 1) / BM;
        int bn = p.N <= 32 ? 32 : (p.N <= 64 ? 64 : (p.N <= 128 ? 128 : 256));
        while (bn > 64 && m_tiles * ((p.N + bn - 1) / bn) < num_sms()) bn /= 2;
        if (bn == 32) return launch_t<32, false, true>(p, s);
        if (bn == 64) return launch_t<64, false, true>(p, s);
        if (bn == 128) return launch_t<128, false, true>(p, s);
        if (use_pair(p)) return launch_pair_t<256, false, true>(p, s);
        return launch_t<256, false, true>(p, s);
    }
    if (use_pair(p)) return launch_pair_t<256, false, false>(p, s);
    // GELU / ReLU first GEMM: 16 epilogue warps while their staging and the
    // segment tables fit in shared memory (up to a few hundred experts)
    if (p.act != 0 && Cfg<256, kEpiWarpsWide>::smem_bytes(p.seg ? p.G : 1) <= (size_t)232448)
        return launch_t<256, false, false, 0, false, false, kEpiWarpsWide>(p, s);
    return launch_t<256, false, false>(p, s);
}

}  // namespace moe
