// landmark_bwd.cu -- gradients of the loss with respect to the landmark
// vectors (sections 1 and 3: the relevance scores take part in next-token
// prediction, so the retriever producing the landmarks learns from the loss;
// rebuttal "Cmt 1": r = sigma l_{c-1} . l_kappa).  For a pool chunk t:
//   dl_t = sigma [ sum_j dr[t+1, j] l_{kappa_{t+1, j}}            (t scores for t+1)
//                + sum_{(c, j) retrieving t} dr[c, j] l_{c-1} ]   (t retrieved)
// One CTA per (batch row, chunk); the second sum walks the inverse retrieval
// index in ascending (query chunk, slot) order, so the result is
// deterministic and no atomics are used.  fp32 accumulation, one chain per
// element in the order above.
// The CTA first stages its list of (landmark row, weight) terms in shared
// memory (the dependent index loads happen once, spread over the threads);
// each thread then owns 16 bytes of the output row and streams the listed
// rows with 16-byte loads that do not depend on one another.  Rows whose size
// is not a multiple of 16 bytes take a scalar kernel.
#include "common.cuh"
#include "kernels.h"

namespace gca {
namespace {

constexpr int kThreads = 256;
constexpr int kVecThreads = 128;
constexpr int kList = 1024;            // terms staged per pass over the list

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

// 16 bytes of a row as fp32 values, and back
__device__ __forceinline__ void unpack16(const uint4& u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4& u, float (&x)[4]) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack16(const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 pack16(const float (&x)[4]) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
}

// Same sums, the row in 16-byte vectors (D * sizeof(T) a multiple of 16).
template <typename T>
__global__ void __launch_bounds__(kVecThreads)
landmark_bwd_vec_kernel(const T* __restrict__ lm, const int32_t* __restrict__ idx,
                        const float* __restrict__ dr, const int* __restrict__ offset,
                        const int* __restrict__ entry, int nC, int D, int topk, float sscale,
                        T* __restrict__ dlm) {
    constexpr int V = 16 / sizeof(T);              // elements per 16-byte vector
    __shared__ int s_r[kList];                     // landmark row of each term (-1: skipped)
    __shared__ float s_w[kList];                   // its d(score)
    const int t = blockIdx.x, b = blockIdx.y;
    const T* row = lm + (size_t)b * nC * D;
    const int* off = offset + (size_t)b * (nC + 1);
    const int* ent = entry + (size_t)b * nC * topk;
    // terms: the top-k slots of chunk t + 1 (t scored them), then the entries
    // (c, j) that retrieved t (t scored by l_{c-1})
    const int n_slot = (t + 1 < nC) ? topk : 0;
    const int e0 = off[t];
    const int n_all = n_slot + (off[t + 1] - e0);
    const int nvec = D / V;
    const int passes = (nvec + kVecThreads - 1) / kVecThreads;
    for (int vp = 0; vp < passes; ++vp) {
        const int v = vp * kVecThreads + threadIdx.x;
        float acc[V];
#pragma unroll
        for (int k = 0; k < V; ++k) acc[k] = 0.f;
        for (int base = 0; base < n_all; base += kList) {
            const int cnt = min(kList, n_all - base);
            __syncthreads();                       // the previous batch has been consumed
            for (int i = threadIdx.x; i < cnt; i += kVecThreads) {
                const int g = base + i;
                int r;
                float w;
                if (g < n_slot) {
                    const size_t q = ((size_t)b * nC + t + 1) * topk + g;
                    r = idx[q];
                    w = dr[q];
                    if (r < 0 || r >= nC) r = -1;
                } else {
                    const int en = ent[e0 + g - n_slot];
                    const int c = en / topk;
                    r = c - 1;
                    w = dr[((size_t)b * nC + c) * topk + en % topk];
                }
                s_r[i] = r;
                s_w[i] = w;
            }
            __syncthreads();
            if (v < nvec) {
                const uint4* src = reinterpret_cast<const uint4*>(row) + v;
                const size_t stride = (size_t)nvec;   // 16-byte vectors per row
#pragma unroll 4
                for (int i = 0; i < cnt; ++i) {
                    const int r = s_r[i];
                    if (r < 0) continue;
                    float x[V];
                    unpack16(__ldg(src + (size_t)r * stride), x);
                    const float w = s_w[i];
#pragma unroll
                    for (int k = 0; k < V; ++k) acc[k] = fmaf(w, x[k], acc[k]);
                }
            }
        }
        if (v < nvec) {
#pragma unroll
            for (int k = 0; k < V; ++k) acc[k] *= sscale;
            reinterpret_cast<uint4*>(dlm + ((size_t)b * nC + t) * D)[v] = pack16(acc);
        }
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
    const size_t esz = p.dtype == GCA_BF16 ? 2 : 4;
    if ((p.D * esz) % 16 == 0) {
        if (p.dtype == GCA_BF16)
            GCA_LAUNCH("landmark_bwd", st,
                       landmark_bwd_vec_kernel<__nv_bfloat16><<<grid, kVecThreads, 0, st>>>(
                           (const __nv_bfloat16*)lm, idx, dscore, offset, entry, p.nQ, p.D, p.topk,
                           p.score_scale, (__nv_bfloat16*)dlm));
        else
            GCA_LAUNCH("landmark_bwd", st,
                       landmark_bwd_vec_kernel<float><<<grid, kVecThreads, 0, st>>>(
                           (const float*)lm, idx, dscore, offset, entry, p.nQ, p.D, p.topk,
                           p.score_scale, (float*)dlm));
    } else if (p.dtype == GCA_BF16)
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
