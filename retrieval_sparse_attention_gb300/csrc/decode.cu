// decode.cu -- decode-time retrieval (sections 3.2 and 4.3 / Table 3 of
// "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling": once per chunk of generated tokens the new
// landmark scores every stored landmark and the top-k chunks are reloaded).
//
// The landmark table is streamed once from HBM in stages of whole rows, dealt
// round-robin to the CTAs (all CTAs read within one moving front of the table);
// each CTA pulls its stages through a shared-memory ring with bulk
// asynchronous copies (cp.async.bulk, one thread issues, an mbarrier counts
// the bytes), so the copy engine keeps HBM busy independently of the math.
// Warps score the staged rows against the query landmark held in registers
// as fp32 (exact for integer landmarks) and keep a running top-k in
// registers, one rank per lane, with the admission threshold replicated in
// every lane so that the common case (row not in the top-k) costs one
// compare.  Merges compare 64-bit rank keys (score, then lower index; keys are
// distinct), so a candidate's place is the number of larger keys among its
// rivals, counted 32 per ballot.  Warps merge into a per-CTA list that way;
// the CTA that finishes last (ticket counter, no waiting) loads every list,
// takes the k-th best list head as a lower bound on the global k-th best (the
// heads are a subset of all rows), keeps the entries ranking at or before it
// (they come from at most topk lists: at most topk^2 of them), ranks those,
// applies the softmax and resets the counter.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "gca_debug.h"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace gca {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBlocks = 2048;
constexpr int kStages = 2;
constexpr int kStageBytes = 49152;
// 64-bit rank keys the last CTA holds in its idle ring: every CTA's list
// (grid * topk) plus room for the survivors of the head bound (at least topk^2)
constexpr int kRingKeys = kStages * kStageBytes / 8;
constexpr int kHeadRegs = 16;            // list heads per lane in the last CTA's registers
constexpr int kMaxGrid = 32 * kHeadRegs; // so at most 512 CTAs

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

struct __align__(8) DecodeBars {
    uint64_t full[kStages], empty[kStages];
    int abort;
    bool is_last;
    unsigned long long bound;      // last CTA: key of the k-th best list head
    int n_kept;                    // last CTA: survivors of the head bound
    unsigned long long top[kMaxTopk];   // merged top-k keys by rank (0: none)
    int stage[kStages];                 // stage held by each slot (-1: no more)
};

template <typename T, int VPL>
__global__ void __launch_bounds__(kThreads)
decode_retrieve_kernel(const T* __restrict__ lm, const T* __restrict__ ql, int N, int D,
                       int topk, int off_by_one, float sscale, int32_t* __restrict__ out_idx,
                       float* __restrict__ out_score, float* __restrict__ out_weight,
                       unsigned* ticket, unsigned* stage_ctr, float* blk_s, int* blk_i,
                       int* status, uint64_t wait_ns, int stall) {
    constexpr int kEPV = 16 / sizeof(T);                 // elements per 16-byte vector
    extern __shared__ uint8_t dsm_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 127) &
                                               ~static_cast<uintptr_t>(127));
    float* qsh = reinterpret_cast<float*>(ring + kStages * kStageBytes);   // [D]
    __shared__ DecodeBars bars;
    __shared__ unsigned long long wkeys[kWarps * kMaxTopk];   // the warps' lists as rank keys

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = D / kEPV;                           // vectors per row (<= 32 * VPL)
    const int row_bytes = nvec * 16;
    const int rows_per_stage = kStageBytes / row_bytes;
    // Stages of the table (rows s*rows_per_stage ...): each CTA's first kStages are
    // dealt round-robin (stage i*grid + cta), later ones are taken from a global
    // counter, so CTAs that run ahead take more and all finish together.
    const int total_stages = (N + rows_per_stage - 1) / rows_per_stage;
    const int dyn0 = kStages * (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&bars.full[i], 1);
            tc::mbar_init(&bars.empty[i], kWarps);
        }
        bars.abort = 0;
        bars.bound = 0ull;
        bars.n_kept = 0;
        tc::fence_barrier_init();
    }
    for (int e = threadIdx.x; e < D; e += kThreads) qsh[e] = to_f(ql[e]);
    __syncthreads();

    // Fill `slot` with stage `sidx` (rows sidx*rows_per_stage ...), or mark it
    // "no more stages" (-1, the full barrier completed without a copy).  Stage
    // indices handed to the slots only grow, so the first -1 ends the CTA's work.
    bool out[kStages] = {};                              // thread 0: copy in flight
    uint32_t oph[kStages] = {};
    auto fill = [&](int slot, int sidx, uint32_t par) {
        if (sidx < total_stages) {
            const int ra = sidx * rows_per_stage;
            const int nr = min(rows_per_stage, N - ra);
            const uint32_t bytes = static_cast<uint32_t>(nr) * row_bytes;
            bars.stage[slot] = sidx;
            tc::mbar_arrive_expect_tx(&bars.full[slot], bytes);
            tcx::bulk_load(ring + slot * kStageBytes,
                           reinterpret_cast<const uint8_t*>(lm) + (size_t)ra * row_bytes, bytes,
                           &bars.full[slot]);
            out[slot] = true;
            oph[slot] = par;
        } else {
            bars.stage[slot] = -1;
            tc::mbar_arrive(&bars.full[slot]);
        }
    };
    int pending = 0;                                     // thread 0: next dynamic stage
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            // fault injection (test only): CTA 0 withholds its first stage, so its
            // bounded waits run out and the timeout path below is taken
            if (stall && blockIdx.x == 0 && i == 0) continue;
            fill(i, i * (int)gridDim.x + (int)blockIdx.x, 0u);
        }
        pending = dyn0 + (int)atomicAdd(stage_ctr, 1u);
    }

    float qv[VPL][kEPV];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const int vi = lane + 32 * u;
#pragma unroll
        for (int x = 0; x < kEPV; ++x) qv[u][x] = (vi < nvec) ? qsh[vi * kEPV + x] : 0.f;
    }

    WarpTopk tk;
    tk.init();
    bool ok = true;
    for (int g = 0;; ++g) {
        const int slot = g % kStages;
        const uint32_t par = static_cast<uint32_t>(g / kStages) & 1u;
        if (!tcx::wait_bar_ns(&bars.abort, &bars.full[slot], par, status, wait_ns)) { ok = false; break; }
        const int sidx = *reinterpret_cast<volatile int*>(&bars.stage[slot]);
        if (threadIdx.x == 0) out[slot] = false;
        if (sidx < 0) break;
        const int ra = sidx * rows_per_stage;
        const int nr = min(rows_per_stage, N - ra);
        const uint4* st = reinterpret_cast<const uint4*>(ring + slot * kStageBytes);
        for (int rr = warp; rr < nr; rr += kWarps) {
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const int vi = lane + 32 * u;
                if (vi < nvec) acc += dot16<T>(st[rr * nvec + vi], qv[u]);
            }
            acc = warp_sum(acc);
            tk.offer(topk, acc, ra + rr);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars.empty[slot]);
        if (threadIdx.x == 0) {
            // refill this slot once every warp has released it
            if (!tcx::wait_bar_ns(&bars.abort, &bars.empty[slot], par, status, wait_ns)) { ok = false; break; }
            const int nxt = pending;
            if (nxt < total_stages) pending = dyn0 + (int)atomicAdd(stage_ctr, 1u);
            fill(slot, nxt, par ^ 1u);
        }
    }
    // Never leave a copy in flight behind an early exit: wait (bounded) for it.
    if (threadIdx.x == 0 && !ok)
        for (int i = 0; i < kStages; ++i)
            if (out[i]) tc::mbar_wait(&bars.full[i], oph[i], nullptr, 100000000ull);

    // CTA merge: every entry of the warps' lists is ranked among all of them
    // by counting larger keys (keys are distinct); ranks below topk are the
    // CTA's list, in order.
    if (lane < topk) wkeys[warp * topk + lane] = tk.ti != 0x7fffffff ? rank_key(tk.ts, tk.ti) : 0ull;
    if (threadIdx.x < kMaxTopk) bars.top[threadIdx.x] = 0ull;
    __syncthreads();
    {
        const int nw = kWarps * topk;
        for (int a = warp; a < nw; a += kWarps) {
            const unsigned long long ka = wkeys[a];
            if (ka == 0ull) continue;
            const int r = warp_rank(ka, wkeys, nw, topk);
            if (r < topk && lane == 0) bars.top[r] = ka;
        }
    }
    __syncthreads();
    if (warp == 0) {
        if (lane < topk) {
            const unsigned long long k = bars.top[lane];
            blk_s[(size_t)blockIdx.x * topk + lane] = k ? key_score(k) : -INFINITY;
            blk_i[(size_t)blockIdx.x * topk + lane] = k ? key_index(k) : 0x7fffffff;
        }
        __threadfence();
        if (lane == 0) bars.is_last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (!bars.is_last) return;

    // Last CTA.  (1) Every CTA's list lands in the idle ring as rank keys.
    // (2) The k-th best of any set of list heads bounds the global k-th best
    // from below (the heads are a subset of all rows); only entries ranking at
    // or before it survive.  The best head of each of 32 lanes gives a cheap
    // bound; if it leaves more survivors than fit, the k-th best of all heads
    // is used, which leaves entries of at most topk lists (topk^2).  (3) The
    // survivors are ranked by counting.
    __threadfence();
    unsigned long long* rk = reinterpret_cast<unsigned long long*>(ring);
    const int nb = gridDim.x;
    const int total = nb * topk;
    unsigned long long* surv = rk + total;
    constexpr int kBatch = 8;       // independent loads in flight per thread
    for (int b0 = threadIdx.x; b0 < total; b0 += kThreads * kBatch) {
        float cs[kBatch];
        int ci[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = b0 + u * kThreads;
            cs[u] = e < total ? __ldcg(blk_s + e) : -INFINITY;
            ci[u] = e < total ? __ldcg(blk_i + e) : 0x7fffffff;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = b0 + u * kThreads;
            if (e < total) rk[e] = ci[u] != 0x7fffffff ? rank_key(cs[u], ci[u]) : 0ull;
        }
    }
    if (threadIdx.x < kMaxTopk) bars.top[threadIdx.x] = 0ull;
    __syncthreads();
    const int cap = kRingKeys - total;                   // survivor room after the lists
    // (2a) cheap bound: the k-th best of the 32 lanes' best heads (a subset of
    // the heads, so still a lower bound on the global k-th best)
    if (warp == 0) {
        unsigned long long best = 0ull;
        for (int c = lane; c < nb; c += 32) {
            const unsigned long long kc = rk[(size_t)c * topk];
            best = kc > best ? kc : best;
        }
        int r = 0;
        for (int o = 0; o < 32; ++o) r += __shfl_sync(0xffffffffu, best, o) > best;
        if (best != 0ull && r == topk - 1) bars.bound = best;
    }
    __syncthreads();
    auto keep_survivors = [&](unsigned long long bound) {
        for (int b0 = warp * 32; b0 < total; b0 += kThreads) {
            const int e = b0 + lane;
            const unsigned long long ke = e < total ? rk[e] : 0ull;
            const bool keep = ke != 0ull && ke >= bound;
            const unsigned m = __ballot_sync(0xffffffffu, keep);
            int base = 0;
            if (lane == 0 && m) base = atomicAdd(&bars.n_kept, __popc(m));
            base = __shfl_sync(0xffffffffu, base, 0);
            const int pos = base + __popc(m & ((1u << lane) - 1u));
            if (keep && pos < cap) surv[pos] = ke;
        }
    };
    keep_survivors(bars.bound);
    __syncthreads();
    if (bars.n_kept > cap) {
        // (2b) too many survivors for the cheap bound: the exact k-th best head
        // bounds them to at most topk lists (topk^2 entries)
        __syncthreads();
        if (threadIdx.x == 0) { bars.n_kept = 0; bars.bound = 0ull; }
        __syncthreads();
        unsigned long long hr[kHeadRegs];      // lane l holds heads l, l + 32, ... (nb <= 32 * kHeadRegs)
#pragma unroll
        for (int j = 0; j < kHeadRegs; ++j) {
            const int c = lane + 32 * j;
            hr[j] = c < nb ? rk[(size_t)c * topk] : 0ull;
        }
        for (int c = warp; c < nb; c += kWarps) {
            const unsigned long long kc = rk[(size_t)c * topk];
            if (kc == 0ull) continue;
            int cnt = 0;
#pragma unroll
            for (int j = 0; j < kHeadRegs; ++j) cnt += hr[j] > kc;
            if (__reduce_add_sync(0xffffffffu, cnt) == topk - 1 && lane == 0) bars.bound = kc;
        }
        __syncthreads();
        keep_survivors(bars.bound);
        __syncthreads();
    }
    const int ns = bars.n_kept;
    for (int a = warp; a < ns; a += kWarps) {
        const unsigned long long ka = surv[a];
        const int r = warp_rank(ka, surv, ns, topk);
        if (r < topk && lane == 0) bars.top[r] = ka;
    }
    __syncthreads();
    if (warp == 0) {
        if (lane < topk && bars.top[lane] != 0ull) {
            tk.ts = key_score(bars.top[lane]);
            tk.ti = key_index(bars.top[lane]);
        } else {
            tk.ts = -INFINITY;
            tk.ti = 0x7fffffff;
        }
        const int m = N < topk ? N : topk;
        const bool okl = lane < m;
        const float r = okl ? tk.ts * sscale : -INFINITY;
        float mx = r;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (off_by_one) mx = fmaxf(mx, 0.f);
        const float e = okl ? expf(r - mx) : 0.f;
        float den = warp_sum(e) + (off_by_one ? expf(-mx) : 0.f);
        if (lane < topk) {
            out_idx[lane] = okl ? tk.ti : -1;
            out_score[lane] = okl ? r : 0.f;
            out_weight[lane] = okl ? e / den : 0.f;
        }
        if (lane == 0) { *ticket = 0u; *stage_ctr = 0u; }     // leave both reset for the next call
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

// Test-only fault injection (gca_debug.h): nonzero = the next decode launch on
// this host thread withholds one stage and bounds its waits by this many ns.
thread_local uint64_t t_stall_wait_ns = 0;

template <typename T, int VPL>
cudaError_t launch_vpl(const void* lm, const void* ql, int N, int D, int topk, int off_by_one,
                       float score_scale, int32_t* idx, float* score, float* weight, void* ws,
                       int* status, cudaStream_t st) {
    auto kern = decode_retrieve_kernel<T, VPL>;
    const size_t smem = (size_t)kStages * kStageBytes + 128 + sizeof(float) * (size_t)D;
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
    // the last CTA holds every list plus topk^2 survivors as keys in its ring
    const int ring_cap = (kRingKeys - topk * topk) / topk;
    if (nb > ring_cap) nb = ring_cap;
    if (nb > kMaxGrid) nb = kMaxGrid;
    float* blk_s = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + 256);
    int* blk_i = reinterpret_cast<int*>(blk_s + (size_t)nb * topk);
    e = cudaMemsetAsync(ticket, 0, 2 * sizeof(unsigned), st);      // ticket and stage counter
    if (e != cudaSuccess) return e;
    const uint64_t stall_ns = t_stall_wait_ns;
    t_stall_wait_ns = 0;
    const uint64_t wait_ns = stall_ns ? stall_ns : tcx::kWaitNs;
    GCA_LAUNCH("decode_retrieve", st,
               kern<<<nb, kThreads, smem, st>>>((const T*)lm, (const T*)ql, N, D, topk, off_by_one,
                                                score_scale, idx, score, weight, ticket, ticket + 1,
                                                blk_s, blk_i, status, wait_ns, stall_ns ? 1 : 0));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const void* lm, const void* ql, int N, int D, int topk, int off_by_one,
                     float sc, int32_t* idx, float* score, float* weight, void* ws, int* status,
                     cudaStream_t st) {
    const int nvec = D * (int)sizeof(T) / 16;
    const int vpl = (nvec + 31) / 32;
    switch (vpl) {
        case 1: return launch_vpl<T, 1>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, status, st);
        case 2: return launch_vpl<T, 2>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, status, st);
        case 3: return launch_vpl<T, 3>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, status, st);
        case 4: return launch_vpl<T, 4>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, status, st);
        case 5: case 6:
            return launch_vpl<T, 6>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, status, st);
        case 7: case 8:
            return launch_vpl<T, 8>(lm, ql, N, D, topk, off_by_one, sc, idx, score, weight, ws, status, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_retrieve(const void* lm, const void* ql, int N, int D, int topk,
                                   gca_dtype_t dt, int off_by_one, float score_scale,
                                   int32_t* idx, float* score, float* weight, void* ws,
                                   int* status, cudaStream_t st, int* launches) {
    cudaError_t e = (dt == GCA_BF16)
        ? launch_t<__nv_bfloat16>(lm, ql, N, D, topk, off_by_one, score_scale, idx, score, weight, ws, status, st)
        : launch_t<float>(lm, ql, N, D, topk, off_by_one, score_scale, idx, score, weight, ws, status, st);
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
void* g_scratch_ptr[kMaxDev];                 // device address of g_decode_scratch per device
unsigned long long g_scratch_ctx[kMaxDev];    // the CUDA context it was looked up in
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device, looked up with
// that device current the first time it is used there (and again if the
// device's context has changed since, e.g. after cudaDeviceReset).  In host
// code the array's name is only a host-side stand-in, never a device address.
cudaError_t static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress((void**)&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();   // the lookup made a context current
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
    int* st = status_word();            // device errors go to the same word as every entry's
    if (!st) return GCA_ERR_CUDA;
    const float sc = score_scale > 0.f ? score_scale : 1.0f / sqrtf((float)D);
    int n = 0;
    const cudaError_t e = launch_decode_retrieve(landmarks, query_landmark, N, D, topk, dtype,
                                                 softmax_off_by_one ? 1 : 0, sc, idx, score,
                                                 weight, ws, st,
                                                 static_cast<cudaStream_t>(stream), &n);
    if (e != cudaSuccess) return GCA_ERR_CUDA;
    set_launch_count(n);
    return GCA_OK;
}

extern "C" gca_status_t gca_debug_stall_next_decode(uint64_t wait_ns) {
    if (wait_ns < 1000ull || wait_ns > 1000000000ull) return GCA_ERR_INVALID_ARG;
    gca::t_stall_wait_ns = wait_ns;
    return GCA_OK;
}
