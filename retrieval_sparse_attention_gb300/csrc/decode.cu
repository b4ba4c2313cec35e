// decode.cu -- decode-time retrieval (sections 3.2 and 4.3 / Table 3 of
// "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling": once per chunk of generated tokens the new
// landmark scores every stored landmark and the top-k chunks are reloaded).
//
// The landmark table is streamed once from HBM: each warp walks rows with
// 16-byte vector loads (several rows in flight), scores them against the
// query landmark held in shared memory as fp32, and keeps a running top-k in
// registers, one rank per lane.  Warps merge into a per-CTA list; the CTA
// that finishes last (ticket counter, no waiting) merges every CTA's list,
// applies the softmax and writes the result.  Scores of integer landmarks
// are exact in fp32, so the ranking is the exact (score desc, index asc) one.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gca {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBlocks = 2048;
constexpr int kRowsInFlight = 4;

// Insert (s, i) into the warp's sorted top-k list (lane j holds rank j).
__device__ __forceinline__ void warp_insert(float& ts, int& ti, int topk, float s, int i) {
    const int lane = threadIdx.x & 31;
    const float ws = __shfl_sync(0xffffffffu, ts, topk - 1);
    const int wi = __shfl_sync(0xffffffffu, ti, topk - 1);
    if (!ranks_before(s, i, ws, wi)) return;            // uniform across the warp
    const unsigned ahead = __ballot_sync(0xffffffffu, lane < topk && ranks_before(ts, ti, s, i));
    const int pos = __popc(ahead);
    const float us = __shfl_up_sync(0xffffffffu, ts, 1);
    const int ui = __shfl_up_sync(0xffffffffu, ti, 1);
    if (lane == pos) { ts = s; ti = i; }
    else if (lane > pos && lane < topk) { ts = us; ti = ui; }
}

template <typename T>
__device__ __forceinline__ float dot16(const uint4& raw, const float* qv);

template <>
__device__ __forceinline__ float dot16<__nv_bfloat16>(const uint4& raw, const float* qv) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float2 f = __bfloat1622float2(h[u]);
        acc = fmaf(f.x, qv[2 * u], acc);
        acc = fmaf(f.y, qv[2 * u + 1], acc);
    }
    return acc;
}

template <>
__device__ __forceinline__ float dot16<float>(const uint4& raw, const float* qv) {
    const float* f = reinterpret_cast<const float*>(&raw);
    return f[0] * qv[0] + f[1] * qv[1] + f[2] * qv[2] + f[3] * qv[3];
}

template <typename T, int VPL>
__global__ void __launch_bounds__(kThreads)
decode_retrieve_kernel(const T* __restrict__ lm, const T* __restrict__ ql, int N, int D,
                       int topk, int off_by_one, float sscale, int32_t* __restrict__ out_idx,
                       float* __restrict__ out_score, float* __restrict__ out_weight,
                       unsigned* ticket, float* blk_s, int* blk_i) {
    constexpr int kEPV = 16 / sizeof(T);                 // elements per 16-byte vector
    extern __shared__ float qsh[];                       // [D] query landmark
    __shared__ float ws_s[kWarps][kMaxTopk];
    __shared__ int ws_i[kWarps][kMaxTopk];
    __shared__ bool is_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < D; e += kThreads) qsh[e] = to_f(ql[e]);
    __syncthreads();

    const int nvec = D / kEPV;                           // vectors per row (<= 32 * VPL)
    float qv[VPL][kEPV];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const int vi = lane + 32 * u;
#pragma unroll
        for (int x = 0; x < kEPV; ++x) qv[u][x] = (vi < nvec) ? qsh[vi * kEPV + x] : 0.f;
    }

    float ts = -INFINITY;
    int ti = 0x7fffffff;
    // Contiguous block of rows per CTA, rows interleaved across its warps.
    const int per_blk = (N + gridDim.x - 1) / gridDim.x;
    const int r0 = blockIdx.x * per_blk;
    const int r1 = min(N, r0 + per_blk);
    const uint4* base = reinterpret_cast<const uint4*>(lm);
    for (int r = r0 + warp * kRowsInFlight; r < r1; r += kWarps * kRowsInFlight) {
        uint4 raw[kRowsInFlight][VPL];
#pragma unroll
        for (int a = 0; a < kRowsInFlight; ++a)
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const int vi = lane + 32 * u;
                if (r + a < r1 && vi < nvec)
                    raw[a][u] = __ldcs(base + (size_t)(r + a) * nvec + vi);
                else
                    raw[a][u] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int a = 0; a < kRowsInFlight; ++a) {
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < VPL; ++u) acc += dot16<T>(raw[a][u], qv[u]);
            acc = warp_sum(acc);
            if (r + a < r1) warp_insert(ts, ti, topk, acc, r + a);
        }
    }
    if (lane < kMaxTopk) { ws_s[warp][lane] = ts; ws_i[warp][lane] = ti; }
    __syncthreads();
    if (warp == 0) {
        for (int w = 1; w < kWarps; ++w)
            for (int j = 0; j < topk; ++j) warp_insert(ts, ti, topk, ws_s[w][j], ws_i[w][j]);
        if (lane < topk) {
            blk_s[(size_t)blockIdx.x * topk + lane] = ts;
            blk_i[(size_t)blockIdx.x * topk + lane] = ti;
        }
        __threadfence();
        if (lane == 0) is_last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;

    // Last CTA: merge every CTA's list (warps split the CTAs, then warp 0).
    __threadfence();
    ts = -INFINITY;
    ti = 0x7fffffff;
    for (int bk = warp; bk < (int)gridDim.x; bk += kWarps)
        for (int j = 0; j < topk; ++j)
            warp_insert(ts, ti, topk, __ldcg(blk_s + (size_t)bk * topk + j),
                        __ldcg(blk_i + (size_t)bk * topk + j));
    if (lane < kMaxTopk) { ws_s[warp][lane] = ts; ws_i[warp][lane] = ti; }
    __syncthreads();
    if (warp == 0) {
        for (int w = 1; w < kWarps; ++w)
            for (int j = 0; j < topk; ++j) warp_insert(ts, ti, topk, ws_s[w][j], ws_i[w][j]);
        const int m = N < topk ? N : topk;
        const bool ok = lane < m;
        const float r = ok ? ts * sscale : -INFINITY;
        float mx = r;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (off_by_one) mx = fmaxf(mx, 0.f);
        const float e = ok ? expf(r - mx) : 0.f;
        float den = warp_sum(e) + (off_by_one ? expf(-mx) : 0.f);
        if (lane < topk) {
            out_idx[lane] = ok ? ti : -1;
            out_score[lane] = ok ? r : 0.f;
            out_weight[lane] = ok ? e / den : 0.f;
        }
        if (lane == 0) *ticket = 0u;     // leave the counter reset for the next call
    }
}

}  // namespace

int decode_max_blocks(int N) {
    int nb = (N + 127) / 128;
    if (nb > kMaxBlocks) nb = kMaxBlocks;
    if (nb < 1) nb = 1;
    return nb;
}

size_t decode_workspace_bytes(int N, int topk) {
    const size_t nb = (size_t)decode_max_blocks(N);
    size_t lists = nb * (size_t)topk * (sizeof(float) + sizeof(int));
    return 256 + ((lists + 255) / 256) * 256;
}

namespace {

template <typename T, int VPL>
cudaError_t launch_vpl(const void* lm, const void* ql, int N, int D, int topk, int off_by_one,
                       float score_scale, int32_t* idx, float* score, float* weight, void* ws,
                       cudaStream_t st) {
    auto kern = decode_retrieve_kernel<T, VPL>;
    const size_t smem = sizeof(float) * (size_t)D;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    int nb = sms * (per_sm > 0 ? per_sm : 1);
    const int cap = decode_max_blocks(N);
    if (nb > cap) nb = cap;
    unsigned* ticket = reinterpret_cast<unsigned*>(ws);
    float* blk_s = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + 256);
    int* blk_i = reinterpret_cast<int*>(blk_s + (size_t)nb * topk);
    e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    GCA_LAUNCH("decode_retrieve", st, kern<<<nb, kThreads, smem, st>>>((const T*)lm, (const T*)ql, N, D, topk, off_by_one,
                                     score_scale, idx, score, weight, ticket, blk_s, blk_i));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const void* lm, const void* ql, int N, int D, int topk, int off_by_one,
                     float sc, int32_t* idx, float* score, float* weight, void* ws, cudaStream_t st) {
    const int nvec = D * (int)sizeof(T) / 16;
    const int vpl = (nvec + 31) / 32;
    switch (vpl) {
        case 1: return launch_vpl<T, 1>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, st);
        case 2: return launch_vpl<T, 2>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, st);
        case 3: return launch_vpl<T, 3>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, st);
        case 4: return launch_vpl<T, 4>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, st);
        case 6: return launch_vpl<T, 6>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, st);
        case 5: case 7: case 8:
            return launch_vpl<T, 8>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_retrieve(const void* lm, const void* ql, int N, int D, int topk,
                                   gca_dtype_t dt, int off_by_one, float score_scale,
                                   int32_t* idx, float* score, float* weight, void* ws,
                                   int* status, cudaStream_t st, int* launches) {
    (void)status;
    cudaError_t e = (dt == GCA_BF16)
        ? launch_t<__nv_bfloat16>(lm, ql, N, D, topk, off_by_one, score_scale, idx, score, weight, ws, st)
        : launch_t<float>(lm, ql, N, D, topk, off_by_one, score_scale, idx, score, weight, ws, st);
    if (e == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace gca

// ---------------------------------------------------------------------------
// Allocation-free variant: the scratch lives in a file-scope device array.
// ---------------------------------------------------------------------------
namespace gca {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[GCA_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device (looked up once
// per device).  In host code the array's name is only a host-side stand-in.
cudaError_t static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace gca

extern "C" gca_status_t gca_decode_retrieve_noalloc(const void* landmarks,
                                                    const void* query_landmark, int N, int D,
                                                    int topk, gca_dtype_t dtype,
                                                    int softmax_off_by_one, float score_scale,
                                                    int32_t* idx, float* score, float* weight,
                                                    void* stream) {
    using namespace gca;
    if (N < 1 || D < 1 || topk < 1) return GCA_ERR_INVALID_ARG;
    if (dtype != GCA_BF16 && dtype != GCA_F32) return GCA_ERR_INVALID_ARG;
    if (!(score_scale >= 0.f)) return GCA_ERR_INVALID_ARG;
    const void* ptrs[5] = {landmarks, query_landmark, idx, score, weight};
    for (const void* p : ptrs)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return GCA_ERR_INVALID_ARG;
    if (topk > kMaxTopk) return GCA_ERR_UNSUPPORTED;
    const int esize = dtype == GCA_BF16 ? 2 : 4;
    if ((D * esize) % 16 != 0 || D * esize > 16 * 256) return GCA_ERR_UNSUPPORTED;
    if (decode_workspace_bytes(N, topk) > GCA_DECODE_STATIC_SCRATCH_BYTES) return GCA_ERR_WORKSPACE;
    void* ws = nullptr;
    if (static_scratch(&ws) != cudaSuccess) return GCA_ERR_CUDA;
    const float sc = score_scale > 0.f ? score_scale : 1.0f / sqrtf((float)D);
    int n = 0;
    const cudaError_t e = launch_decode_retrieve(landmarks, query_landmark, N, D, topk, dtype,
                                                 softmax_off_by_one ? 1 : 0, sc, idx, score,
                                                 weight, ws, nullptr,
                                                 static_cast<cudaStream_t>(stream), &n);
    return e == cudaSuccess ? GCA_OK : GCA_ERR_CUDA;
}
