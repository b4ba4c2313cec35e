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

// One thread per (b, c): reduce the partial dw (per head and per quarter of
// the chunk's tokens) in a fixed order, then
// apply the softmax Jacobian (same form for the vanilla and off-by-one
// softmax, whose Jacobians are both diag(w) - w w^T).
__global__ void dscore_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w,
                              const float* __restrict__ dwpart, int n_rows, int H, int topk,
                              int nP, float* __restrict__ dscore) {
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= n_rows) return;
    float dw[kMaxTopk];
    float wdw = 0.f;
    for (int j = 0; j < topk; ++j) {
        float acc = 0.f;
        for (int hq = 0; hq < 4 * H; ++hq) acc += dwpart[((size_t)row * 4 * H + hq) * topk + j];
        dw[j] = acc;
        const int kap = idx[(size_t)row * topk + j];
        if (kap >= 0 && kap < nP) wdw += w[(size_t)row * topk + j] * acc;
    }
    for (int j = 0; j < topk; ++j) {
        const size_t o = (size_t)row * topk + j;
        const int kap = idx[o];
        dscore[o] = (kap >= 0 && kap < nP) ? w[o] * (dw[j] - wdw) : 0.f;
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
    GCA_LAUNCH("dscore", st, dscore_kernel<<<(rows + 127) / 128, 128, 0, st>>>(idx, w, dwpart, rows, s.H, s.topk, s.nP, dscore));
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace gca
