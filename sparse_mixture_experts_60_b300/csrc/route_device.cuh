// Device helpers of the routing step shared by the router kernels
// (router.cu) and the routing epilogue of the tensor-core router GEMM
// (gemm_sm103.cu).  Pages: "MoE Training: Mixture of Experts" (Quick Start
// MoELayer: softmax, topk, renormalise); "Mixture of Experts (MoE) From
// Scratch to DeepSeek V3" (sigmoid routing with selection bias b_i).
#pragma once

#include <math.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- fp32 key
// The sigmoid selection key must be reproducible bit for bit, so it is a
// fixed sequence of correctly rounded fp32 operations (explicit _rn
// intrinsics: no contraction, no reassociation):
//   exp: Cody-Waite reduction n = rint(a log2e), r = a - n ln2 with ln 2
//        split into a 16-bit head (exact products) and an fp32 tail, then
//        the degree-7 Taylor polynomial of e^r in Horner form, then one
//        multiply by the exact power of two 2^n;  a > 88 -> +inf,
//        a < -87 -> 0.
//   sigmoid(x) = 1 / (1 + exp(-x));  key = sigmoid(logit) + b_i.
__device__ __forceinline__ float exp_key(float a) {
    if (a != a) return a;
    if (a > 88.0f) return __int_as_float(0x7f800000);
    if (a < -87.0f) return 0.0f;
    const float n = rintf(__fmul_rn(a, 0x1.715476p+0f));
    float r = __fmaf_rn(-n, 0x1.62e4p-1f, a);
    r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
    float q = 0x1.a01a02p-13f;           // 1/7!
    q = __fmaf_rn(q, r, 0x1.6c16c2p-10f);  // 1/6!
    q = __fmaf_rn(q, r, 0x1.111112p-7f);   // 1/5!
    q = __fmaf_rn(q, r, 0x1.555556p-5f);   // 1/4!
    q = __fmaf_rn(q, r, 0x1.555556p-3f);   // 1/3!
    q = __fmaf_rn(q, r, 0x1p-1f);          // 1/2!
    q = __fmaf_rn(q, r, 1.0f);
    q = __fmaf_rn(q, r, 1.0f);
    const int ni = (int)n;                 // -126 .. 127
    return __fmul_rn(q, __int_as_float((ni + 127) << 23));
}

__device__ __forceinline__ float sigmoid_key(float x) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_key(-x)));
}

// (key descending, expert ascending)
__device__ __forceinline__ bool ranks_before(float ka, int ea, float kb, int eb) {
    return ka > kb || (ka == kb && ea < eb);
}

// After the loop, lane l holds the warp-wide sum of v[l] (a reduce-scatter
// by recursive halving: 31 shuffles for 32 values).
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

// Route one token whose E <= EP logits are l[0..E) of this thread (one
// thread per token; EP = 8, 16 or 32 bounds every loop).  Keys are the
// logits (softmax routing) or sigmoid_key(logit) + b_i (sigmoid routing);
// the k largest keys are taken in k arg-max rounds (equal keys: lower
// expert index), each round recording its expert's rank and gate in
// per-expert registers.  Gates are the softmax probabilities (or sigmoid
// scores) of the chosen experts, renormalised over the k when asked.  For a
// valid token writes topk_idx/topk_w [k] at t*k and lse[t]; returns the
// chosen experts as a bit mask and the logsumexp in *lse_out.
template <int EP>
__device__ __forceinline__ uint32_t route_row(const float (&l)[EP], int E, int k, int score_fn, int renormalize,
                                              const float *sel_bias, bool valid, int64_t t, int32_t *topk_idx,
                                              float *topk_w, float *lse_arr, float *lse_out) {
    float key[EP];
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
        float kv = -INFINITY;
        if (e < E) {
            kv = score_fn == 0 ? l[e] : __fadd_rn(sigmoid_key(l[e]), sel_bias ? __ldg(sel_bias + e) : 0.0f);
            if (kv != kv) kv = -INFINITY;
            m = fmaxf(m, l[e]);
        }
        key[e] = kv;
    }
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < EP; ++e)
        if (e < E) s += expf(l[e] - m);
    const float lse = m + logf(s);
    *lse_out = lse;
    int rank[EP];
    float gsel[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) {
        rank[e] = -1;
        gsel[e] = 0.0f;
    }
    uint32_t taken = 0u;
    float tot = 0.0f;
    for (int j = 0; j < k; ++j) {
        float bk = -INFINITY, bl = 0.0f;
        int be = 0;
        bool any = false;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            if (e < E && !((taken >> e) & 1u) && (!any || ranks_before(key[e], e, bk, be))) {
                bk = key[e];
                be = e;
                bl = l[e];
                any = true;
            }
        }
        taken |= 1u << be;
        const float g = score_fn == 0 ? expf(bl - m) : 1.0f / (1.0f + expf(-bl));
        tot += g;
#pragma unroll
        for (int e = 0; e < EP; ++e)
            if (e == be) {
                rank[e] = j;
                gsel[e] = g;
            }
    }
    if (valid) {
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            if (rank[e] >= 0) {
                float w;
                if (renormalize) w = gsel[e] / tot;
                else w = score_fn == 0 ? expf(l[e] - lse) : gsel[e];
                topk_idx[t * k + rank[e]] = e;
                topk_w[t * k + rank[e]] = w;
            }
        }
        lse_arr[t] = lse;
    }
    return valid ? taken : 0u;
}

}  // namespace moe
