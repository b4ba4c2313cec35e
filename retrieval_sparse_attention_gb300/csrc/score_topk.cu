// score_topk.cu -- causal relevance scoring fused with top-k and the weight
// softmax (rebuttal "Cmt 1": Eq. 1 with one group, r = l_t^T l_k / sqrt(d);
// README "Model Architecture": the landmark of chunk c-1 selects the chunks
// that chunk c attends to; rebuttal Q4: Eq. 3 is the softmax off by one).
//
// One CTA per (batch row, query chunk).  The landmark of chunk c-1 is staged
// in shared memory as fp32; each warp scores a strided subset of the earlier
// chunks, two at a time (lanes split D in 16-byte vectors, fp32 FMA,
// warp-shuffle sum: exact for integer landmarks with |s| < 2^24) and keeps a
// running top-k of its keys in registers under the order (score descending,
// chunk ascending); the eight warp lists are merged by counting, for each
// entry, the entries ranking before it.  The whole landmark tensor of a row
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
#include "topk.cuh"

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
    float* s = sh + D;         // [nC]  clean scores of the candidates
    __shared__ float sel_s[kMaxTopk];
    __shared__ int sel_i[kMaxTopk];
    __shared__ unsigned long long wkeys[kWarps * kMaxTopk];   // the warps' lists as rank keys
    __shared__ unsigned long long top[kMaxTopk];               // merged list by rank

    const int c = blockIdx.x, b = blockIdx.y;
    const int t = c - 1;
    const int n = (t < 0) ? 0 : (include_self ? t + 1 : t);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* row = lm + (size_t)b * nC * D;

    if (t >= 0)
        for (int e = threadIdx.x; e < D; e += kThreads) lt[e] = to_f(row[(size_t)t * D + e]);
    __syncthreads();

    // scores: a warp per candidate, two candidates in flight (16-byte loads of
    // the candidate rows when D allows it); each warp keeps a running top-k of
    // the selection keys it produced, in registers
    constexpr int kEPV = 16 / sizeof(T);
    const bool vec = (D % kEPV) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const float* nrow = NOISY ? noise + ((size_t)b * nC + c) * nC : nullptr;
    WarpTopk tk;
    tk.init();
    auto record = [&](int kap, float acc) {
        const float kv = NOISY ? __fadd_rn(__fmul_rn(acc, sscale), nrow[kap]) : acc;
        if (lane == 0) s[kap] = acc;
        tk.offer(topk, kv, kap);
    };
    for (int k0 = warp; k0 < n; k0 += 2 * kWarps) {
        const int k1 = k0 + kWarps;
        float a0 = 0.f, a1 = 0.f;
        if (vec) {
            const uint4* r0 = reinterpret_cast<const uint4*>(row + (size_t)k0 * D);
            const uint4* r1 = reinterpret_cast<const uint4*>(row + (size_t)(k1 < n ? k1 : k0) * D);
            const float4* l4 = reinterpret_cast<const float4*>(lt);
            for (int v = lane; v < D / kEPV; v += 32) {
                const uint4 x0 = __ldg(r0 + v), x1 = __ldg(r1 + v);
                const T* e0 = reinterpret_cast<const T*>(&x0);
                const T* e1 = reinterpret_cast<const T*>(&x1);
#pragma unroll
                for (int w4 = 0; w4 < kEPV / 4; ++w4) {
                    const float4 q = l4[v * (kEPV / 4) + w4];
                    const float qa[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        a0 = fmaf(qa[u], to_f(e0[4 * w4 + u]), a0);
                        a1 = fmaf(qa[u], to_f(e1[4 * w4 + u]), a1);
                    }
                }
            }
        } else {
            const T* r0 = row + (size_t)k0 * D;
            const T* r1 = row + (size_t)(k1 < n ? k1 : k0) * D;
            for (int e = lane; e < D; e += 32) {
                a0 = fmaf(lt[e], to_f(r0[e]), a0);
                a1 = fmaf(lt[e], to_f(r1[e]), a1);
            }
        }
        record(k0, warp_sum(a0));
        const float s1 = warp_sum(a1);
        if (k1 < n) record(k1, s1);
    }

    // merge the warps' lists: an entry's place is the number of larger rank
    // keys among all entries (keys are distinct), counted 32 per ballot
    if (lane < topk) wkeys[warp * topk + lane] = tk.ti != 0x7fffffff ? rank_key(tk.ts, tk.ti) : 0ull;
    if (threadIdx.x < kMaxTopk) top[threadIdx.x] = 0ull;
    __syncthreads();
    const int m = n < topk ? n : topk;
    {
        const int nw = kWarps * topk;
        for (int a = warp; a < nw; a += kWarps) {
            const unsigned long long ka = wkeys[a];
            if (ka == 0ull) continue;
            const int r = warp_rank(ka, wkeys, nw, topk);
            if (r < topk && lane == 0) top[r] = ka;
        }
    }
    __syncthreads();
    if (threadIdx.x < m) {
        const int kap = key_index(top[threadIdx.x]);
        sel_i[threadIdx.x] = kap;
        sel_s[threadIdx.x] = s[kap];       // the clean score
    }
    __syncthreads();

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
    const size_t smem = sizeof(float) * ((size_t)sp.D + (size_t)sp.nQ);
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
    if (score_topk_tc_supported(sp)) {
        // bf16 landmarks with D a multiple of 64: scores from the tensor cores
        const cudaError_t e = launch_score_topk_tc(sp, lm, noise, idx, score, weight, status, st);
        if (e == cudaSuccess) *launches += 1;
        return e;
    }
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
