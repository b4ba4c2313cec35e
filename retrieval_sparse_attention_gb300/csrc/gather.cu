// gather.cu -- reload of retrieved chunks from an offloaded K/V cache
// (section 3.2 and the rebuttal's offload estimate: past chunks' key/value
// representations can live in CPU memory and be brought back only when
// retrieved, G times every S tokens).
//
// The cache is [n_chunks, chunk_bytes] in memory the GPU can address: device
// memory, or page-locked host memory (with unified addressing its host
// pointer is valid on the device and is read over the CPU-GPU link).  The
// retrieved chunks of K and of V are streamed with 16-byte loads into a
// compact device pool [topk, chunk], and each slot's new index (j, or -1 for
// an empty slot) is written, so that gca_fwd can run on the compact pool.
// Each chunk is split over many CTAs, each issuing all its loads before its
// stores, so the link's latency is paid about once per call.
#include "common.cuh"
#include "kernels.h"

namespace gca {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

__global__ void __launch_bounds__(kThreads)
gather_chunks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                     int n_src, size_t chunk_vecs, const int32_t* __restrict__ idx, int topk,
                     uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                     int32_t* __restrict__ dst_idx, int* status) {
    const int j = blockIdx.x;
    const int kap = idx[j];
    const bool ok = kap >= 0 && kap < n_src;
    if (threadIdx.x == 0 && blockIdx.y == 0) {
        dst_idx[j] = ok ? j : -1;
        if (kap >= n_src) set_status(status, GCA_ERR_DEVICE_INDEX);
    }
    // this CTA's piece: kThreads * kUnroll vectors of the chunk's K and of its V,
    // every load issued before any store (the link's latency is paid once)
    const size_t base = (size_t)blockIdx.y * kThreads * kUnroll + threadIdx.x;
    const uint4 z = make_uint4(0, 0, 0, 0);
    const uint4* sk = src_k + (size_t)(ok ? kap : 0) * chunk_vecs;
    const uint4* sv = src_v + (size_t)(ok ? kap : 0) * chunk_vecs;
    uint4 a[kUnroll], c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const size_t i = base + (size_t)u * kThreads;
        a[u] = (ok && i < chunk_vecs) ? __ldcs(sk + i) : z;
        c[u] = (ok && i < chunk_vecs) ? __ldcs(sv + i) : z;
    }
    uint4* dk = dst_k + (size_t)j * chunk_vecs;
    uint4* dv = dst_v + (size_t)j * chunk_vecs;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const size_t i = base + (size_t)u * kThreads;
        if (i < chunk_vecs) {
            dk[i] = a[u];
            dv[i] = c[u];
        }
    }
}

}  // namespace

cudaError_t launch_gather_chunks(const void* src_k, const void* src_v, int n_src, size_t chunk_bytes,
                                 const int32_t* idx, int topk, void* dst_k, void* dst_v,
                                 int32_t* dst_idx, int* status, cudaStream_t st, int* launches) {
    const size_t vecs = chunk_bytes / 16;
    // one CTA per kThreads * kUnroll vectors of a chunk: the whole transfer is
    // in flight at once for chunks of the usual size
    const size_t per_cta = (size_t)kThreads * kUnroll;
    const size_t split = (vecs + per_cta - 1) / per_cta;
    if (split < 1 || split > 65535) return cudaErrorInvalidValue;
    dim3 grid(topk, (unsigned)split);
    GCA_LAUNCH("gather_chunks", st,
               gather_chunks_kernel<<<grid, kThreads, 0, st>>>(
                   (const uint4*)src_k, (const uint4*)src_v, n_src, vecs, idx, topk, (uint4*)dst_k,
                   (uint4*)dst_v, dst_idx, status));
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace gca
