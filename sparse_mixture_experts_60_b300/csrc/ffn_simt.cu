// Grouped expert FFN layer for fp32 storage on the CUDA cores.
//
// Same contract as the tensor-core grouped GEMM (rows seg[g]..seg[g+1]-1 of
// A against the weights of group g, bias + GELU/ReLU or SwiGLU gating in the
// epilogue), in full fp32: the fp32 layer is the small exact-precision
// case, and tf32 tensor cores would not hold its 1e-4 relative tolerance.
//
// Pages: "MoE Training: Mixture of Experts" (Quick Start expert);
// "moe_code.py" (Expert, FFN(x) = ReLU(x W1 + b1) W2 + b2).
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <bool GATED>
__global__ void __launch_bounds__(256) ffn_simt_kernel(SimtProblem p) {
    PDL_ENTER();
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN + 4];
    __shared__ float B2s[GATED ? TK : 1][TN + 4];
    const int g = blockIdx.z;
    const int64_t seg0 = p.seg ? p.seg[g] : 0;
    const int64_t rows = p.seg ? (int64_t)p.seg[g + 1] - seg0 : p.M;
    const int64_t r0 = (int64_t)blockIdx.y * TM;
    if (r0 >= rows) return;
    const int n0 = blockIdx.x * TN;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {}, acc2[4][4] = {};
    const float *Bg = p.B + (int64_t)g * p.N * p.K;
    const float *B2g = GATED ? p.B2 + (int64_t)g * p.N * p.K : nullptr;
    for (int k0 = 0; k0 < p.K; k0 += TK) {
        for (int i = threadIdx.x; i < TM * TK; i += 256) {
            const int r = i / TK, kk = i % TK;
            const int64_t row = r0 + r;
            const int kc = k0 + kk;
            As[kk][r] = (row < rows && kc < p.K) ? p.A[(seg0 + row) * p.K + kc] : 0.0f;
            const int n = n0 + r;
            Bs[kk][r] = (n < p.N && kc < p.K) ? Bg[(int64_t)n * p.K + kc] : 0.0f;
            if (GATED) B2s[kk][r] = (n < p.N && kc < p.K) ? B2g[(int64_t)n * p.K + kc] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float a[4], b[4], b2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
                if (GATED) b2[i] = B2s[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if (GATED) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = r0 + ty * 4 + i;
        if (row >= rows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= p.N) continue;
            float v = acc[i][j];
            if (GATED) {
                v = v / (1.0f + expf(-v)) * acc2[i][j];
            } else {
                if (p.bias) v += p.bias[(int64_t)g * p.bias_stride + n];
                if (p.act == 1) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
                else if (p.act == 2) v = fmaxf(v, 0.0f);
            }
            p.out[(seg0 + row) * p.ldo + n] = v;
        }
    }
}

}  // namespace

cudaError_t launch_ffn_simt(const SimtProblem &p, cudaStream_t s) {
    const int G = p.seg ? p.G : 1;
    const int64_t max_rows = p.seg ? p.max_rows : p.M;
    if (max_rows <= 0 || G <= 0) return cudaSuccess;
    dim3 grid((unsigned)ceil_div(p.N, TN), (unsigned)ceil_div(max_rows, TM), (unsigned)G);
    if (p.gated) return launch_pdl(ffn_simt_kernel<true>, grid, dim3(256), 0, s, p);
    return launch_pdl(ffn_simt_kernel<false>, grid, dim3(256), 0, s, p);
}

}  // namespace moe
