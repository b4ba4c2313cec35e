// bwd_common.cu -- pieces of the GCA backward shared by both element types:
// the backward workspace layout, the inverse retrieval index that lets the
// key-major pass visit every (query chunk, slot) that retrieved a pool chunk
// in a fixed order, and the relevance-score gradient
//   dr_j = w_j (dw_j - sum_i w_i dw_i),  dw_j = sum over the chunk's tokens
//   and heads of dO_t . O_t^j
// (App. B backward: gradients for the weights; section 3: the scores learn
// from the next-token loss through the fusion weights).
#include "common.cuh"
#include "kernels.h"

namespace gca {

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

BwdWorkspace bwd_workspace_layout(const Shape& s) {
    BwdWorkspace w{};
    size_t off = 0;
    w.delta_off = off;  off += align256(sizeof(float) * (size_t)s.B * s.Lq * s.H * s.topk);
    w.dwpart_off = off; off += align256(sizeof(float) * (size_t)s.B * s.nQ * s.H * 4 * s.topk);
    w.lse2_off = off;   off += align256(sizeof(float) * (size_t)s.B * s.Lq * s.H * s.topk);
    w.count_off = off;  off += align256(sizeof(int) * (size_t)s.B * s.nP);
    w.offset_off = off; off += align256(sizeof(int) * (size_t)s.B * (s.nP + 1));
    w.entry_off = off;  off += align256(sizeof(int) * (size_t)s.B * s.nQ * s.topk);
    w.entry_w_off = off; off += align256(sizeof(float) * (size_t)s.B * s.nQ * s.topk);
    w.order_off = off;  off += align256(sizeof(int) * (size_t)s.B * s.nP);
    w.total = off;
    return w;
}

namespace {

constexpr int kWarpsPerBlock = 8;

// One warp per (b, kappa): count the entries of idx[b] equal to kappa.
__global__ void inv_count_kernel(const int32_t* __restrict__ idx, int B, int nE, int nP,
                                 int* __restrict__ count) {
    const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= B * nP) return;
    const int b = gw / nP, kap = gw % nP;
    const int32_t* row = idx + (size_t)b * nE;
    int n = 0;
    for (int e0 = 0; e0 < nE; e0 += 32) {
        const int e = e0 + lane;
        const bool hit = e < nE && row[e] == kap;
        n += __popc(__ballot_sync(0xffffffffu, hit));
    }
    if (lane == 0) count[gw] = n;
}

// One CTA per batch row: exclusive prefix sum of the counts into offsets.
__global__ void inv_scan_kernel(const int* __restrict__ count, int nP, int* __restrict__ offset) {
    __shared__ int part[1024];
    const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    const int per = (nP + nt - 1) / nt;
    const int lo = min(nP, tid * per), hi = min(nP, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += count[(size_t)b * nP + i];
    part[tid] = sum;
    __syncthreads();
    for (int o = 1; o < nt; o <<= 1) {           // Hillis-Steele inclusive scan
        int v = tid >= o ? part[tid - o] : 0;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    int run = part[tid] - sum;
    int* off = offset + (size_t)b * (nP + 1);
    for (int i = lo; i < hi; ++i) { off[i] = run; run += count[(size_t)b * nP + i]; }
    if (tid == nt - 1) off[nP] = part[nt - 1];
}

// One warp per (b, kappa): write the entries e = c*topk + j with
// idx[b][e] == kappa, in ascending e, into the CSR bucket of kappa (and, if
// entry_w is given, the weight w[b][e] beside each, so that a reader of the
// bucket needs no dependent load).
__global__ void inv_fill_kernel(const int32_t* __restrict__ idx, int B, int nE, int nP,
                                const int* __restrict__ offset, int* __restrict__ entry,
                                const float* __restrict__ w, float* __restrict__ entry_w) {
    const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= B * nP) return;
    const int b = gw / nP, kap = gw % nP;
    const int32_t* row = idx + (size_t)b * nE;
    int* out = entry + (size_t)b * nE;
    int pos = offset[(size_t)b * (nP + 1) + kap];
    const unsigned below = (1u << lane) - 1u;
    for (int e0 = 0; e0 < nE; e0 += 32) {
        const int e = e0 + lane;
        const bool hit = e < nE && row[e] == kap;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit) {
            const int at = pos + __popc(m & below);
            out[at] = e;
            if (entry_w) entry_w[(size_t)b * nE + at] = w[(size_t)b * nE + e];
        }
        pos += __popc(m);
    }
}

// One warp per (b, c): lane l sums the partials (head, token quarter) l, l + 32, ... of
// every slot, a shuffle tree over the warp (fixed order, lane 0's result broadcast)
// gives the slot totals dw_j, then the softmax Jacobian (same form for the vanilla
// and off-by-one softmax, whose Jacobians are both diag(w) - w w^T):
// dr_j = w_j (dw_j - sum_i w_i dw_i).
__global__ void dscore_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w,
                              const float* __restrict__ dwpart, int n_rows, int H, int topk,
                              int nP, float* __restrict__ dscore) {
    const int row = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= n_rows) return;
    const float* dp = dwpart + (size_t)row * 4 * H * topk;
    float acc[kMaxTopk];
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) acc[j] = 0.f;
    for (int hq = lane; hq < 4 * H; hq += 32) {
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j)
            if (j < topk) acc[j] += dp[(size_t)hq * topk + j];
    }
    float wdw = 0.f, mine = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
        if (j >= topk) break;
        float v = acc[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
        v = __shfl_sync(0xffffffffu, v, 0);
        if (lane == j) mine = v;
        const int kap = idx[(size_t)row * topk + j];
        if (kap >= 0 && kap < nP) wdw += w[(size_t)row * topk + j] * v;
    }
    if (lane < topk) {
        const size_t o = (size_t)row * topk + lane;
        const int kap = idx[o];
        dscore[o] = (kap >= 0 && kap < nP) ? w[o] * (mine - wdw) : 0.f;
    }
}

// The whole inverse index of one batch row in one CTA (a stable counting sort of
// the row's entries by retrieved chunk).  The row's idx is staged in shared
// memory and cut into one contiguous segment per warp.  (1) Each warp counts its
// segment per chunk: lanes that hold the same chunk form a __match_any_sync
// group whose highest lane adds the group size (each warp owns its count row:
// no atomics).  (2) Per chunk, the warps' counts become exclusive prefixes over
// the warps, and the chunk totals are scanned into offsets.  (3) Each warp places
// its segment in ascending entry order: slot = offset + its warps' prefix + rank in
// the group.  (4) The CTA writes the entries out, each with its weight.
__global__ void inv_index_kernel(const int32_t* __restrict__ idx, int nE, int nP, int nw,
                                 int* __restrict__ count, int* __restrict__ offset,
                                 int* __restrict__ entry, const float* __restrict__ w,
                                 float* __restrict__ entry_w) {
    extern __shared__ int sh[];
    int* ent = sh;                          // [nE]: the row's idx
    int* fill = sh + nE;                    // [nE]: the entries in bucket order
    int* off = sh + 2 * nE;                 // [nP + 1]: bucket offsets
    int* wc = sh + 2 * nE + nP + 1;         // [nw][nP]: per-warp counts, then prefixes
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* row = idx + (size_t)b * nE;
    const int seg = ((nE + nw - 1) / nw + 31) / 32 * 32;
    for (int i = tid; i < nw * nP; i += blockDim.x) wc[i] = 0;
    for (int e = tid; e < nE; e += blockDim.x) ent[e] = row[e];
    __syncthreads();
    const unsigned below = (1u << lane) - 1u;
    if (warp < nw) {
        int* mine = wc + (size_t)warp * nP;
        for (int e0 = warp * seg; e0 < min(nE, (warp + 1) * seg); e0 += 32) {
            const int e = e0 + lane;
            const int k = e < nE ? ent[e] : -1;
            const bool valid = k >= 0 && k < nP;
            const unsigned grp = __match_any_sync(0xffffffffu, valid ? k : -1);
            if (valid && lane == 31 - __clz(grp)) mine[k] += __popc(grp);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int k = tid; k < nP; k += blockDim.x) {      // per chunk: prefix over the warps
        int run = 0;
        for (int v = 0; v < nw; ++v) {
            const int c = wc[(size_t)v * nP + k];
            wc[(size_t)v * nP + k] = run;
            run += c;
        }
        off[k] = run;                                 // the chunk's total, scanned below
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < nP; base += 32) {
            const int i = base + lane;
            const int v = i < nP ? off[i] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (i < nP) {
                count[(size_t)b * nP + i] = v;
                off[i] = run + incl - v;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) off[nP] = run;
    }
    __syncthreads();
    for (int i = tid; i <= nP; i += blockDim.x) offset[(size_t)b * (nP + 1) + i] = off[i];
    if (warp < nw) {
        int* mine = wc + (size_t)warp * nP;
        for (int e0 = warp * seg; e0 < min(nE, (warp + 1) * seg); e0 += 32) {
            const int e = e0 + lane;
            const int k = e < nE ? ent[e] : -1;
            const bool valid = k >= 0 && k < nP;
            const unsigned grp = __match_any_sync(0xffffffffu, valid ? k : -1);
            if (valid) fill[off[k] + mine[k] + __popc(grp & below)] = e;
            __syncwarp();
            if (valid && lane == 31 - __clz(grp)) mine[k] += __popc(grp);
            __syncwarp();
        }
    }
    __syncthreads();
    const int n = off[nP];
    for (int i = tid; i < n; i += blockDim.x) {
        const int e = fill[i];
        entry[(size_t)b * nE + i] = e;
        if (entry_w) entry_w[(size_t)b * nE + i] = w[(size_t)b * nE + e];
    }
}

}  // namespace

cudaError_t launch_inverse_index(const Shape& s, const int32_t* idx, const float* w, void* ws,
                                 cudaStream_t st, int* launches) {
    const BwdWorkspace L = bwd_workspace_layout(s);
    char* base = static_cast<char*>(ws);
    return launch_inverse_index_to(s, idx, reinterpret_cast<int*>(base + L.count_off),
                                   reinterpret_cast<int*>(base + L.offset_off),
                                   reinterpret_cast<int*>(base + L.entry_off), w,
                                   reinterpret_cast<float*>(base + L.entry_w_off), st, launches);
}

size_t inverse_index_bytes(int B, int nQ, int nP, int topk) {
    return align256(sizeof(int) * (size_t)B * nP) + align256(sizeof(int) * (size_t)B * (nP + 1)) +
           align256(sizeof(int) * (size_t)B * nQ * topk);
}

cudaError_t launch_inverse_index_to(const Shape& s, const int32_t* idx, int* count, int* offset,
                                    int* entry, const float* w, float* entry_w, cudaStream_t st,
                                    int* launches) {
    const int nE = s.nQ * s.topk;
    // one CTA per row while its staging fits shared memory (a CTA may use 227 KB):
    // 32 warps' count rows for up to 512 chunks, 8 for more (16 measured slower at
    // 1024 chunks: the per-chunk prefix over the warps grows with them).  The
    // three-pass fallback scans the whole row once per chunk, so it is only for
    // rows that do not fit.
    const int nw = s.nP <= 512 ? 32 : 8;
    const size_t smem = sizeof(int) * (2 * (size_t)nE + (size_t)s.nP + 1 + (size_t)nw * s.nP);
    if (smem <= 220 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(inv_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        GCA_LAUNCH("inv_index", st, inv_index_kernel<<<s.B, 1024, smem, st>>>(idx, nE, s.nP, nw, count, offset,
                                                                               entry, w, w ? entry_w : nullptr));
        *launches += 1;
        return cudaGetLastError();
    }
    // rows too long for one CTA's shared memory: count, scan and fill as three passes
    const int warps = s.B * s.nP;
    const int blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    GCA_LAUNCH("inv_count", st, inv_count_kernel<<<blocks, 32 * kWarpsPerBlock, 0, st>>>(idx, s.B, nE, s.nP, count));
    GCA_LAUNCH("inv_scan", st, inv_scan_kernel<<<s.B, 1024, 0, st>>>(count, s.nP, offset));
    GCA_LAUNCH("inv_fill", st, inv_fill_kernel<<<blocks, 32 * kWarpsPerBlock, 0, st>>>(idx, s.B, nE, s.nP, offset, entry,
                                                                                   w, w ? entry_w : nullptr));
    *launches += 3;
    return cudaGetLastError();
}

cudaError_t launch_dscore(const Shape& s, const int32_t* idx, const float* w, void* ws,
                          float* dscore, cudaStream_t st, int* launches) {
    const BwdWorkspace L = bwd_workspace_layout(s);
    const float* dwpart = reinterpret_cast<const float*>(static_cast<char*>(ws) + L.dwpart_off);
    const int rows = s.B * s.nQ;
    GCA_LAUNCH("dscore", st, dscore_kernel<<<(rows + kWarpsPerBlock - 1) / kWarpsPerBlock, 32 * kWarpsPerBlock, 0, st>>>(
                                 idx, w, dwpart, rows, s.H, s.topk, s.nP, dscore));
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace gca
