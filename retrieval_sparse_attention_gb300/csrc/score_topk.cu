// score_topk.cu -- causal relevance scoring fused with top-k and the weight
// softmax (rebuttal "Cmt 1": Eq. 1 with one group, r = l_t^T l_k / sqrt(d);
// README "Model Architecture": the landmark of chunk c-1 selects the chunks
// that chunk c attends to; rebuttal Q4: Eq. 3 is the softmax off by one).
//
// One CTA per (batch row, query chunk).  The landmark of chunk c-1 is staged
// in shared memory as fp32; each warp scores a strided subset of the earlier
// chunks (lanes split D, fp32 FMA, warp-shuffle sum: exact for integer
// landmarks with |s| < 2^24), the scores stay in shared memory, and the
// top-k is taken by k rounds of a block-wide arg-max under the order
// (score descending, chunk ascending).  The whole landmark tensor of a row
// is small (nC x D) and stays in L2, so the kernel is latency-bound.
//
// With a noise tensor (section 3.2: during training Gumbel noise is added to
// the relevance scores before the top-k selection) the selection key is
// fl32(fl32(s * sigma) + g), rounded step by step; the weights are still the
// softmax of the clean scores of the selected chunks.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gca {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T, bool NOISY>
__global__ void __launch_bounds__(kThreads)
score_topk_kernel(const T* __restrict__ lm, const float* __restrict__ noise, int nC, int D,
                  int topk, int include_self, int off_by_one, float sscale,
                  int32_t* __restrict__ idx, float* __restrict__ score,
                  float* __restrict__ weight) {
    extern __shared__ float sh[];
    float* lt = sh;            // [D]   landmark of chunk c-1
    float* s = sh + D;         // [nC]  scores of the candidates
    float* key = NOISY ? s + nC : s;   // [nC] selection keys
    __shared__ float red_s[kWarps];
    __shared__ int red_i[kWarps];
    __shared__ float sel_s[kMaxTopk];
    __shared__ int sel_i[kMaxTopk];

    const int c = blockIdx.x, b = blockIdx.y;
    const int t = c - 1;
    const int n = (t < 0) ? 0 : (include_self ? t + 1 : t);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* row = lm + (size_t)b * nC * D;

    if (t >= 0)
        for (int e = threadIdx.x; e < D; e += kThreads) lt[e] = to_f(row[(size_t)t * D + e]);
    __syncthreads();

    for (int kap = warp; kap < n; kap += kWarps) {
        const T* lk = row + (size_t)kap * D;
        float acc = 0.f;
        for (int e = lane; e < D; e += 32) acc = fmaf(lt[e], to_f(lk[e]), acc);
        acc = warp_sum(acc);
        if (lane == 0) {
            s[kap] = acc;
            if (NOISY)
                key[kap] = __fadd_rn(__fmul_rn(acc, sscale),
                                     noise[((size_t)b * nC + c) * nC + kap]);
        }
    }
    __syncthreads();

    const int m = n < topk ? n : topk;
    for (int j = 0; j < m; ++j) {
        float bs = -INFINITY;
        int bi = 0x7fffffff;
        for (int kap = threadIdx.x; kap < n; kap += kThreads) {
            float v = key[kap];
            if (v != -INFINITY && ranks_before(v, kap, bs, bi)) { bs = v; bi = kap; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float os = __shfl_xor_sync(0xffffffffu, bs, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_before(os, oi, bs, bi)) { bs = os; bi = oi; }
        }
        if (lane == 0) { red_s[warp] = bs; red_i[warp] = bi; }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kWarps; ++w)
                if (ranks_before(red_s[w], red_i[w], bs, bi)) { bs = red_s[w]; bi = red_i[w]; }
            sel_s[j] = s[bi];    // the clean score
            sel_i[j] = bi;
            key[bi] = -INFINITY; // taken
        }
        __syncthreads();
    }

    if (threadIdx.x == 0) {
        const size_t o = ((size_t)b * nC + c) * topk;
        float r[kMaxTopk];
        float mx = -INFINITY;
        for (int j = 0; j < m; ++j) { r[j] = sel_s[j] * sscale; mx = fmaxf(mx, r[j]); }
        if (off_by_one) mx = fmaxf(mx, 0.f);
        float den = off_by_one ? expf(-mx) : 0.f;
        for (int j = 0; j < m; ++j) den += expf(r[j] - mx);
        for (int j = 0; j < topk; ++j) {
            const bool ok = j < m;
            idx[o + j] = ok ? sel_i[j] : -1;
            score[o + j] = ok ? r[j] : 0.f;
            weight[o + j] = ok ? expf(r[j] - mx) / den : 0.f;
        }
    }
}

template <typename T, bool NOISY>
void launch_typed(const Shape& sp, const void* lm, const float* noise, int32_t* idx, float* score,
                  float* weight, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((size_t)sp.D + (NOISY ? 2 : 1) * (size_t)sp.nQ);
    dim3 grid(sp.nQ, sp.B);
    auto kern = score_topk_kernel<T, NOISY>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    GCA_LAUNCH(NOISY ? "score_topk_noisy" : "score_topk", st,
               kern<<<grid, kThreads, smem, st>>>((const T*)lm, noise, sp.nQ, sp.D, sp.topk,
                                                  sp.include_self, sp.off_by_one, sp.score_scale,
                                                  idx, score, weight));
}

}  // namespace

cudaError_t launch_score_topk(const Shape& sp, const void* lm, const float* noise, int32_t* idx,
                              float* score, float* weight, int* status, cudaStream_t st,
                              int* launches) {
    (void)status;
    if (sp.dtype == GCA_BF16) {
        if (noise) launch_typed<__nv_bfloat16, true>(sp, lm, noise, idx, score, weight, st);
        else launch_typed<__nv_bfloat16, false>(sp, lm, noise, idx, score, weight, st);
    } else {
        if (noise) launch_typed<float, true>(sp, lm, noise, idx, score, weight, st);
        else launch_typed<float, false>(sp, lm, noise, idx, score, weight, st);
    }
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace gca
