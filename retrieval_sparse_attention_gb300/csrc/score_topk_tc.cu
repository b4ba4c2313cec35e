// score_topk_tc.cu -- causal relevance scoring, top-k and weight softmax with
// the scores from the tensor cores (bf16 landmarks, D a multiple of 64).
//
// The relevance of candidate chunk kappa for query chunk c is
// s = l_{c-1} . l_kappa (rebuttal "Cmt 1": Eq. 1 with one group; README "Model
// Architecture": the landmark of chunk c-1 selects the chunks chunk c attends
// to), i.e. one entry of the Gram matrix L L^T of a batch row's landmarks.
// A cluster of kCL CTAs owns 128 consecutive landmark rows t (query chunks
// c = t + 1); CTA rank r of the cluster computes their Gram-matrix entries
// against the r-th of kCL equal slices (a multiple of 16 candidates) of the
// tile's candidate range, in candidate tiles of up to 128: TMA stages 64-column
// blocks of the row tile and of the candidate tile (128-byte swizzle), one
// thread issues tcgen05.mma (M = 128, N = the tile width, bf16 products, fp32
// accumulation over the K blocks in order: exact for integer landmarks with
// |s| < 2^24, and every entry is summed whole inside one CTA) into up to four
// TMEM accumulators, and four epilogue threads per row t read the row's scores
// from TMEM and keep running top-k lists in registers, offered in ascending
// candidate order, so ties keep the lower chunk index (score descending, then
// chunk ascending).  The four lists of a row are merged through shared memory;
// then, after a cluster barrier, each CTA merges 128 / kCL rows' lists from all
// kCL CTAs of the cluster (distributed shared memory: the slices are disjoint
// and ordered) and computes the softmax (vanilla or off by one, rebuttal Q4)
// of the selected scores.  A second cluster barrier keeps every CTA's lists in
// place until all have been read.  Nothing is written but idx / score /
// weight, so no workspace is needed.
//
// With a noise tensor (section 3.2: Gumbel noise added to the relevance
// scores before the top-k selection) the selection key is
// fl32(fl32(s * sigma) + g), rounded step by step; the weights are the softmax
// of the clean scores of the selected chunks.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace gca {
namespace {

using namespace tc;

// warp 0 producer, warp 1 MMA issuer, warps 4-19 epilogue: four threads per
// landmark row, each owning a quarter of every candidate tile's columns
constexpr int kThreads = 640;
constexpr int kEpi = 512;
constexpr int kRows = 128;             // landmark rows per CTA (and per candidate tile)
constexpr int kBlk = 64;               // landmark columns per stage block
constexpr int kStages = 6;
constexpr int kTile = kRows * kBlk * 2;          // one 128 x 64 bf16 tile, 16 KB
constexpr int kStageBytes = 2 * kTile;           // row tile block, then candidate tile block
constexpr int kAcc = 4;                          // candidate tiles accumulated at once (4 x 128 TMEM columns)
constexpr int kSmem = kStages * kStageBytes + 1024;
// the epilogue's four lists per row (key, clean score, chunk) reuse the stages,
// followed by the row's merged list that the cluster reads
static_assert(3 * kRows * 5 * 16 * 4 + 3 * kRows * 16 * 4 <= kStages * kStageBytes, "list merge area");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives, then waits: release/acquire
// order the shared-memory lists written before it with the reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of this CTA's shared-memory word `p` in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

struct __align__(8) GramBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full, acc_empty;
    uint64_t done;
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

// Element of a candidate list: selection key, clean score (differs from the key
// only with noise), chunk.  Lists are sorted by (key descending, chunk
// ascending); an empty entry is (-inf, 0, 0x7fffffff) and ranks last.
struct Cand {
    float k, s;
    int i;
};
__device__ __forceinline__ bool ranks_first(const Cand& a, const Cand& b) {
    return a.k > b.k || (a.k == b.k && a.i < b.i);
}
// Compare-exchange: afterwards a ranks first.  Branch-free selects, so every
// lane runs the same instructions and the networks below have no data-dependent
// control flow.
template <bool WITH_S>
__device__ __forceinline__ void cex(Cand& a, Cand& b) {
    const bool sw = ranks_first(b, a);
    const Cand t = a;
    a.k = sw ? b.k : a.k;
    a.i = sw ? b.i : a.i;
    b.k = sw ? t.k : b.k;
    b.i = sw ? t.i : b.i;
    if (WITH_S) {
        a.s = sw ? b.s : a.s;
        b.s = sw ? t.s : b.s;
    }
}
// Bitonic sort of N (a power of two) elements into rank order.
template <int N, bool WITH_S>
__device__ __forceinline__ void bitonic_sort(Cand (&c)[N]) {
#pragma unroll
    for (int k = 2; k <= N; k *= 2)
#pragma unroll
        for (int j = k / 2; j > 0; j /= 2)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    if ((i & k) == 0) cex<WITH_S>(c[i], c[l]);
                    else cex<WITH_S>(c[l], c[i]);
                }
            }
}
// Bitonic sequence of N elements -> rank order.
template <int N, bool WITH_S>
__device__ __forceinline__ void bitonic_clean(Cand (&c)[N]) {
#pragma unroll
    for (int j = N / 2; j > 0; j /= 2)
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int l = i ^ j;
            if (l > i) cex<WITH_S>(c[i], c[l]);
        }
}

// Running top-KCAP of one thread (KCAP >= the call's k, so the first k entries
// are its top-k).  A chunk of 16 (or 8) candidates is sorted by a bitonic
// network and merged: the better of list[i] and chunk[KCAP - 1 - i] for every i is exactly
// the top KCAP of the union, as a bitonic sequence, which a half-cleaner cascade
// puts in order.  No insertion chain, no run-time index into the list (which
// would move it out of registers).
template <int KCAP, bool WITH_S>
struct RowTopk {
    Cand e[KCAP];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int p = 0; p < KCAP; ++p) e[p] = Cand{-INFINITY, 0.f, 0x7fffffff};
    }
    // merge N (8 or 16) candidates; with N < KCAP the chunk is padded with empty
    // entries, which never win, so only its N real entries are compared
    template <int N>
    __device__ __forceinline__ void merge(Cand (&c)[N]) {
        bitonic_sort<N, WITH_S>(c);
#pragma unroll
        for (int p = 0; p < KCAP; ++p)
            if (KCAP - 1 - p < N && ranks_first(c[KCAP - 1 - p < N ? KCAP - 1 - p : 0], e[p]))
                e[p] = c[KCAP - 1 - p < N ? KCAP - 1 - p : 0];
        bitonic_clean<KCAP, WITH_S>(e);
    }
};

// kCL = CTAs per cluster = candidate slices per row tile (4 or 8)
template <int KCAP, bool NOISY, int kCL>
__global__ void __launch_bounds__(kThreads, 1)
score_topk_tc_kernel(const __grid_constant__ CUtensorMap tl, const float* __restrict__ noise, int nC,
                     int D, int topk, int include_self, int off_by_one, float sscale,
                     int32_t* __restrict__ idx, float* __restrict__ score, float* __restrict__ weight,
                     int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ GramBars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int crank = static_cast<int>(cluster_rank());
    const int R = blockIdx.x / kCL, b = blockIdx.y;
    const int row0 = R * kRows;
    // the tile's candidates are the chunks below its last row; this CTA takes the
    // slice [c_lo, c_hi) in tiles of up to 128 candidates (tile j starts at c_lo + 128 j)
    const int range = min((R + 1) * kRows, nC);
    const int span = 16 * ((range + 16 * kCL - 1) / (16 * kCL));
    const int c_lo = min(crank * span, range), c_hi = min(c_lo + span, range);
    const int ntile = (c_hi - c_lo + kRows - 1) / kRows;
    // MMA width of tile j: its candidates rounded up to 16 (columns past c_hi are ignored)
    auto tile_n = [&](int j) { return min(kRows, (c_hi - c_lo - j * kRows + 15) & ~15); };
    const int nkb = D / kBlk;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, status); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sb.full[i], 1);
            mbar_init(&sb.empty[i], 1);
        }
        mbar_init(&sb.acc_full, 1);
        mbar_init(&sb.acc_empty, kEpi);
        mbar_init(&sb.done, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tl);
    if (warp == 1) {
        tmem_alloc(&sb.tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    if (warp == 0) {
        if (lane == 0) {
            tcx::Ring st{0, 0};
            bool out[kStages] = {};
            uint32_t oph[kStages] = {};
            bool ok = true;
            for (int c0 = 0; c0 < ntile && ok; c0 += kAcc) {
                const int nj = min(kAcc, ntile - c0);
                for (int kb = 0; kb < nkb && ok; ++kb) {
                    for (int j = 0; j < nj; ++j) {
                        if (!wait(&sb.empty[st.i], st.ph ^ 1u)) { ok = false; break; }
                        uint8_t* stg = sm + st.i * kStageBytes;
                        mbar_arrive_expect_tx(&sb.full[st.i], kStageBytes);
                        tma_load_3d(stg, &tl, &sb.full[st.i], kb * kBlk, row0, b);
                        tma_load_3d(stg + kTile, &tl, &sb.full[st.i], kb * kBlk, c_lo + (c0 + j) * kRows, b);
                        out[st.i] = true;
                        oph[st.i] = st.ph;
                        st.next(kStages);
                    }
                }
            }
            for (int i = 0; i < kStages; ++i)
                if (out[i]) mbar_wait(&sb.full[i], oph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            tcx::Ring st{0, 0};
            bool ok = true, issued = false;
            int chunk = 0;
            for (int c0 = 0; c0 < ntile && ok; c0 += kAcc, ++chunk) {
                const int nj = min(kAcc, ntile - c0);
                // the epilogue has read the previous chunk's accumulators
                if (!wait(&sb.acc_empty, empty_par(chunk))) break;
                tc_fence_after();
                for (int kb = 0; kb < nkb && ok; ++kb) {
                    for (int j = 0; j < nj; ++j) {
                        if (!wait(&sb.full[st.i], st.ph)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a = smem_u32(sm + st.i * kStageBytes);
                        const uint32_t id = idesc_bf16(128, tile_n(c0 + j), false, false);
                        tcx::mma_kmajor_k64(tmem + j * 128, a, a + kTile, id, kb > 0 ? 1u : 0u);
                        mma_commit(&sb.empty[st.i]);
                        issued = true;
                        st.next(kStages);
                    }
                }
                if (ok) mma_commit(&sb.acc_full);
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp >= 4) {
        // epilogue: thread (r, cq) owns landmark row t = row0 + r (query chunk c = t + 1)
        // and columns 32 cq .. 32 cq + 31 of every candidate tile
        const int qd = warp & 3, cq = (warp - 4) >> 2;
        const int r = 32 * qd + lane;
        const int t = row0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        // candidates kappa < t (kappa <= t with include_self) for c = t + 1 <= nC - 1
        const int lim = (t + 1 <= nC - 1) ? (include_self ? t + 1 : t) : 0;
        const float* nrow = NOISY ? noise + ((size_t)b * nC + (t + 1 < nC ? t + 1 : 0)) * nC : nullptr;
        RowTopk<KCAP, NOISY> tk;
        tk.init();
        bool ok = true;
        int chunk = 0;
        for (int c0 = 0; c0 < ntile; c0 += kAcc, ++chunk) {
            const int nj = min(kAcc, ntile - c0);
            if (!wait(&sb.acc_full, full_par(chunk))) { ok = false; break; }
            tc_fence_after();
            for (int j = 0; j < nj; ++j) {
                const int kap0 = c_lo + (c0 + j) * kRows + 32 * cq;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    if (32 * cq + 16 * q >= tile_n(c0 + j)) break;     // warp-uniform: no such columns
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tmem + lane_base + j * 128 + 32 * cq + 16 * q, v);
                    tmem_wait_ld();
                    const int k16 = kap0 + 16 * q;
                    // the candidates of these columns in chunks of CW (invalid ones rank
                    // last); skip a chunk when no lane has one that beats its list's last
                    // entry.  k <= 16 with noise merges halves of 8: 16 + 16 entries of
                    // three fields would not fit the registers.
                    constexpr int CW = (KCAP == 16 && NOISY) ? 8 : 16;
#pragma unroll
                    for (int h0 = 0; h0 < 16; h0 += CW) {
                        Cand c[CW];
                        bool any = false;
#pragma unroll
                        for (int u = 0; u < CW; ++u) {
                            const int kap = k16 + h0 + u;
                            const float sc = __uint_as_float(v[h0 + u]);
                            const bool in = kap < lim && kap < c_hi;
                            const float kv = (NOISY && in) ? __fadd_rn(__fmul_rn(sc, sscale), __ldg(nrow + kap)) : sc;
                            c[u] = in ? Cand{kv, sc, kap} : Cand{-INFINITY, 0.f, 0x7fffffff};
                            any = any || (in && ranks_first(c[u], tk.e[KCAP - 1]));
                        }
                        if (__any_sync(0xffffffffu, any)) tk.template merge<CW>(c);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sb.acc_empty);
        }
        // merge the four lists of each row through the stage memory (every product
        // that read it has completed: the last accumulators were full), into the
        // row's list that the other CTAs of the cluster read
        float* lk = reinterpret_cast<float*>(sm);                 // [128 rows][4][KCAP] keys
        float* ls = lk + kRows * 4 * KCAP;                         // clean scores
        int* li = reinterpret_cast<int*>(ls + kRows * 4 * KCAP);   // chunks
        float* mk = reinterpret_cast<float*>(li + kRows * 4 * KCAP);   // [128 rows][KCAP] merged
        float* ms = mk + kRows * KCAP;
        int* mi = reinterpret_cast<int*>(ms + kRows * KCAP);
        const int base = (r * 4 + cq) * KCAP;
#pragma unroll
        for (int p = 0; p < KCAP; ++p) { lk[base + p] = tk.e[p].k; ls[base + p] = NOISY ? tk.e[p].s : tk.e[p].k; li[base + p] = tk.e[p].i; }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpi) : "memory");
        if (cq == 0) {
            // four sorted lists of disjoint candidates (entries past a list's end are
            // -inf / no chunk): take the best head KCAP times
            int h[4] = {0, 0, 0, 0};
            const int rb = r * 4 * KCAP;
#pragma unroll
            for (int j = 0; j < KCAP; ++j) {
                int best = -1, bi = 0x7fffffff;
                float bk = -INFINITY, bs = 0.f;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const bool in = h[qq] < KCAP;
                    const int at = rb + qq * KCAP + (in ? h[qq] : 0);
                    const float kq = in ? lk[at] : -INFINITY;
                    const int iq = in ? li[at] : 0x7fffffff;
                    if (iq != 0x7fffffff && (best < 0 || kq > bk || (kq == bk && iq < bi))) {
                        best = qq; bk = kq; bi = iq; bs = ls[at];
                    }
                }
                mk[r * KCAP + j] = bk;
                ms[r * KCAP + j] = bs;
                mi[r * KCAP + j] = bi;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) h[qq] += (best == qq) ? 1 : 0;
            }
        }
    }

    // every thread of the cluster: the merged lists are complete
    cluster_sync();
    // rows kRowsPer crank .. of the tile (128 / kCL of them): warps 4-7 first copy
    // the lists of the kCL CTAs into this CTA's shared memory (128 threads, one
    // (row, CTA) list each, independent loads), then one thread per row merges them
    constexpr int kRowsPer = kRows / kCL;
    {
        float* mk = reinterpret_cast<float*>(sm) + 3 * kRows * 4 * KCAP;
        float* ms = mk + kRows * KCAP;
        int* mi = reinterpret_cast<int*>(ms + kRows * KCAP);
        // local copies [kRowsPer rows][kCL][KCAP] after this CTA's own lists (which the
        // other CTAs may still be reading)
        float* ck = reinterpret_cast<float*>(mi + kRows * KCAP);
        float* cs = ck + kRowsPer * kCL * KCAP;
        int* ci = reinterpret_cast<int*>(cs + kRowsPer * kCL * KCAP);
        if (warp >= 4 && warp < 8) {
            const int tid = threadIdx.x - 128;
            const int rl = tid / kCL, q = tid % kCL;
            const int at = (kRowsPer * crank + rl) * KCAP;
            const uint32_t rk = map_rank(mk + at, q), rs = map_rank(ms + at, q), ri = map_rank(mi + at, q);
            uint32_t vk[KCAP], vs[KCAP], vi[KCAP];
#pragma unroll
            for (int p = 0; p < KCAP; ++p) {
                vk[p] = ld_cluster_u32(rk + 4 * p);
                vs[p] = ld_cluster_u32(rs + 4 * p);
                vi[p] = ld_cluster_u32(ri + 4 * p);
            }
            const int lb = (rl * kCL + q) * KCAP;
#pragma unroll
            for (int p = 0; p < KCAP; ++p) {
                ck[lb + p] = __uint_as_float(vk[p]);
                cs[lb + p] = __uint_as_float(vs[p]);
                ci[lb + p] = static_cast<int>(vi[p]);
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");
        }
        if (warp == 4 && lane < kRowsPer) {
            const int r = kRowsPer * crank + lane;
            const int t = row0 + r;
            if (t + 1 <= nC - 1) {
                const int lim = include_self ? t + 1 : t;
                int h[kCL];
#pragma unroll
                for (int q = 0; q < kCL; ++q) h[q] = 0;
                Cand mg[KCAP];
                const int rb = lane * kCL * KCAP;
#pragma unroll
                for (int j = 0; j < KCAP; ++j) {
                    if (j < topk) {
                        // the CTAs' candidate slices are in rank order: equal keys keep the lower chunk
                        int best = -1, bi = 0x7fffffff;
                        float bk = -INFINITY, bs = 0.f;
#pragma unroll
                        for (int q = 0; q < kCL; ++q) {
                            const bool in = h[q] < KCAP;
                            const int at = rb + q * KCAP + (in ? h[q] : 0);
                            const int iq = in ? ci[at] : 0x7fffffff;
                            const float kq = in ? ck[at] : -INFINITY;
                            if (iq != 0x7fffffff && (best < 0 || kq > bk || (kq == bk && iq < bi))) {
                                best = q; bk = kq; bi = iq; bs = cs[at];
                            }
                        }
                        mg[j] = Cand{bk, bs, bi};
#pragma unroll
                        for (int q = 0; q < kCL; ++q) h[q] += (best == q) ? 1 : 0;
                    }
                }
                const size_t o = ((size_t)b * nC + t + 1) * topk;
                const int m = lim < topk ? lim : topk;
                float rr[KCAP];
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < KCAP; ++j) {
                    rr[j] = (j < m) ? mg[j].s * sscale : -INFINITY;
                    mx = fmaxf(mx, rr[j]);
                }
                if (off_by_one) mx = fmaxf(mx, 0.f);
                float den = off_by_one ? expf(-mx) : 0.f;
#pragma unroll
                for (int j = 0; j < KCAP; ++j)
                    if (j < m) den += expf(rr[j] - mx);
#pragma unroll
                for (int j = 0; j < KCAP; ++j) {
                    if (j < topk) {
                        const bool v = j < m;
                        idx[o + j] = v ? mg[j].i : -1;
                        score[o + j] = v ? rr[j] : 0.f;
                        weight[o + j] = v ? expf(rr[j] - mx) / den : 0.f;
                    }
                }
            }
            if (R == 0 && crank == 0 && lane == 0) {
                // query chunk 0 has no earlier chunk to retrieve
                const size_t o = (size_t)b * nC * topk;
                for (int j = 0; j < topk; ++j) { idx[o + j] = -1; score[o + j] = 0.f; weight[o + j] = 0.f; }
            }
        }
    }
    // no CTA leaves while another may still read its lists
    cluster_sync();

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int KCAP, bool NOISY, int CL>
cudaError_t launch_cl(const Shape& sp, const CUtensorMap& tl, const float* noise, int32_t* idx,
                      float* score, float* weight, int* status, cudaStream_t st) {
    auto kern = score_topk_tc_kernel<KCAP, NOISY, CL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * ((sp.nQ + kRows - 1) / kRows), sp.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    GCA_LAUNCH(NOISY ? "score_topk_noisy" : "score_topk", st,
               e = cudaLaunchKernelEx(&cfg, kern, tl, noise, sp.nQ, sp.D, sp.topk, sp.include_self,
                                      sp.off_by_one, sp.score_scale, idx, score, weight, status));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Clusters of 8 while the whole grid stays within 64 CTAs (measured: 128 CTAs in
// clusters of 8 ran in two waves, slower than 64 in clusters of 4), else 4.
template <int KCAP, bool NOISY>
cudaError_t launch_k(const Shape& sp, const CUtensorMap& tl, const float* noise, int32_t* idx,
                     float* score, float* weight, int* status, cudaStream_t st) {
    const int tiles = sp.B * ((sp.nQ + kRows - 1) / kRows);
    if (tiles * 8 <= 64) return launch_cl<KCAP, NOISY, 8>(sp, tl, noise, idx, score, weight, status, st);
    return launch_cl<KCAP, NOISY, 4>(sp, tl, noise, idx, score, weight, status, st);
}

}  // namespace

// bf16 landmarks with D a multiple of 64 and k <= 16 (the lists per row live in
// registers; larger k runs the SIMT scorer).
bool score_topk_tc_supported(const Shape& sp) {
    return sp.dtype == GCA_BF16 && sp.D % kBlk == 0 && sp.D <= 8192 && sp.nQ >= 2 && sp.topk <= 16;
}

cudaError_t launch_score_topk_tc(const Shape& sp, const void* lm, const float* noise, int32_t* idx,
                                 float* score, float* weight, int* status, cudaStream_t st) {
    CUtensorMap tl;
    // [B, nC, D] as sequences: rows past a batch row's nC read as zeros
    if (!encode_bf16_seq(&tl, lm, sp.B, sp.nQ, sp.D, kRows)) return cudaErrorInvalidValue;
    const bool nz = noise != nullptr;
    if (sp.topk <= 8) return nz ? launch_k<8, true>(sp, tl, noise, idx, score, weight, status, st)
                                : launch_k<8, false>(sp, tl, noise, idx, score, weight, status, st);
    return nz ? launch_k<16, true>(sp, tl, noise, idx, score, weight, status, st)
              : launch_k<16, false>(sp, tl, noise, idx, score, weight, status, st);
}

}  // namespace gca
