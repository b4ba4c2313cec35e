// landmark_bwd.cu -- gradients of the loss with respect to the landmark
// vectors (sections 1 and 3: the relevance scores take part in next-token
// prediction, so the retriever producing the landmarks learns from the loss;
// rebuttal "Cmt 1": r = sigma l_{c-1} . l_kappa).  For a pool chunk t:
//   dl_t = sigma [ sum_j dr[t+1, j] l_{kappa_{t+1, j}}            (t scores for t+1)
//                + sum_{(c, j) retrieving t} dr[c, j] l_{c-1} ]   (t retrieved)
// One CTA per (batch row, chunk); the second sum walks the inverse retrieval
// index in ascending (query chunk, slot) order, so the result is
// deterministic and no atomics are used.  fp32 accumulation.
#include "common.cuh"
#include "kernels.h"

namespace gca {
namespace {

constexpr int kThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kThreads)
landmark_bwd_kernel(const T* __restrict__ lm, const int32_t* __restrict__ idx,
                    const float* __restrict__ dr, const int* __restrict__ offset,
                    const int* __restrict__ entry, int nC, int D, int topk, float sscale,
                    T* __restrict__ dlm) {
    const int t = blockIdx.x, b = blockIdx.y;
    const T* row = lm + (size_t)b * nC * D;
    const int nE = nC * topk;
    const int* off = offset + (size_t)b * (nC + 1);
    const int* ent = entry + (size_t)b * nE;
    for (int e = threadIdx.x; e < D; e += kThreads) {
        float acc = 0.f;
        if (t + 1 < nC) {
            const size_t r0 = ((size_t)b * nC + t + 1) * topk;
            for (int j = 0; j < topk; ++j) {
                const int kap = idx[r0 + j];
                if (kap < 0 || kap >= nC) continue;
                acc = fmaf(dr[r0 + j], to_f(row[(size_t)kap * D + e]), acc);
            }
        }
        for (int n = off[t]; n < off[t + 1]; ++n) {
            const int en = ent[n];
            const int c = en / topk;
            acc = fmaf(dr[((size_t)b * nC + c) * topk + en % topk], to_f(row[(size_t)(c - 1) * D + e]),
                       acc);
        }
        dlm[((size_t)b * nC + t) * D + e] = from_f<T>(acc * sscale);
    }
}

}  // namespace

cudaError_t launch_landmark_bwd(const Shape& s, const void* lm, const int32_t* idx,
                                const float* dscore, void* dlm, void* ws, cudaStream_t st,
                                int* launches) {
    // the pool of a landmark row is its own chunks
    Shape p = s;
    p.nP = s.nQ;
    char* base = static_cast<char*>(ws);
    int* count = reinterpret_cast<int*>(base);
    const size_t c_bytes = ((sizeof(int) * (size_t)p.B * p.nP) + 255) / 256 * 256;
    int* offset = reinterpret_cast<int*>(base + c_bytes);
    const size_t o_bytes = ((sizeof(int) * (size_t)p.B * (p.nP + 1)) + 255) / 256 * 256;
    int* entry = reinterpret_cast<int*>(base + c_bytes + o_bytes);
    cudaError_t e = launch_inverse_index_to(p, idx, count, offset, entry, nullptr, nullptr, st, launches);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nQ, p.B);
    if (p.dtype == GCA_BF16)
        GCA_LAUNCH("landmark_bwd", st,
                   landmark_bwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
                       (const __nv_bfloat16*)lm, idx, dscore, offset, entry, p.nQ, p.D, p.topk,
                       p.score_scale, (__nv_bfloat16*)dlm));
    else
        GCA_LAUNCH("landmark_bwd", st,
                   landmark_bwd_kernel<float><<<grid, kThreads, 0, st>>>(
                       (const float*)lm, idx, dscore, offset, entry, p.nQ, p.D, p.topk,
                       p.score_scale, (float*)dlm));
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace gca
