// score_topk_tc.cu -- causal relevance scoring, top-k and weight softmax with
// the scores from the tensor cores (bf16 landmarks, D a multiple of 64).
//
// The relevance of candidate chunk kappa for query chunk c is
// s = l_{c-1} . l_kappa (rebuttal "Cmt 1": Eq. 1 with one group; README "Model
// Architecture": the landmark of chunk c-1 selects the chunks chunk c attends
// to), i.e. one entry of the Gram matrix L L^T of a batch row's landmarks.
// One CTA owns 128 consecutive landmark rows t (query chunks c = t + 1) and
// computes their rows of the Gram matrix tile by tile: TMA stages 64-column
// blocks of the row tile and of a 128-row candidate tile (128-byte swizzle),
// one thread issues tcgen05.mma (M = 128, N = 128, bf16 products, fp32
// accumulation: exact for integer landmarks with |s| < 2^24) into up to four
// TMEM accumulators, and each of 128 epilogue threads owns one row t: it reads
// the row's scores from TMEM and keeps a running top-k of them in registers
// (four threads per row, each over a quarter of the columns; their lists are
// merged at the end),
// offered in ascending candidate order, so ties keep the lower chunk index
// (score descending, then chunk ascending).  The softmax (vanilla or off by
// one, rebuttal Q4) of the selected scores is computed by the same thread.
// Nothing is written but idx / score / weight, so no workspace is needed.
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
// the epilogue's four lists per row (key, clean score, chunk) reuse the stages
static_assert(3 * kRows * 4 * 16 * 4 <= kStages * kStageBytes, "list merge area");

struct __align__(8) GramBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full, acc_empty;
    uint64_t done;
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

// Running top-k of one thread, sorted by (key descending, chunk ascending);
// candidates arrive in ascending chunk order, so a candidate whose key equals
// the k-th key ranks after it and is rejected.
template <int KCAP>
struct RowTopk {
    float key[KCAP];       // selection key (the score, or the noisy key)
    float s[KCAP];         // clean score
    int i[KCAP];
    float thr;             // key of rank topk - 1
    bool full;             // topk entries held
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int p = 0; p < KCAP; ++p) { key[p] = -INFINITY; s[p] = 0.f; i[p] = 0x7fffffff; }
        thr = -INFINITY;
        full = false;
    }
    // Insert (kv, sc, ix); kv = -inf with ix = 0x7fffffff is a no-op.  Branch-free,
    // so the lanes of a warp insert in lock step.
    __device__ __forceinline__ void insert(int topk, float kv, float sc, int ix) {
        // one insertion pass: the carried entry swaps with every entry it ranks before
        float ck = kv, cs = sc;
        int ci = ix;
#pragma unroll
        for (int p = 0; p < KCAP; ++p) {
            if (p < topk) {
                const bool before = ck > key[p] || (ck == key[p] && ci < i[p]);
                const float tk = key[p], ts = s[p];
                const int ti = i[p];
                key[p] = before ? ck : tk;
                s[p] = before ? cs : ts;
                i[p] = before ? ci : ti;
                ck = before ? tk : ck;
                cs = before ? ts : cs;
                ci = before ? ti : ci;
            }
            if (p == topk - 1) {
                thr = key[p];
                full = i[p] != 0x7fffffff;
            }
        }
    }
};

template <int KCAP, bool NOISY>
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
    const int R = blockIdx.x, b = blockIdx.y;
    const int row0 = R * kRows;
    // candidate tiles 0 .. R hold every chunk below this tile's last row
    const int ntile = R + 1;
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
                        tma_load_3d(stg + kTile, &tl, &sb.full[st.i], kb * kBlk, (c0 + j) * kRows, b);
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
            const uint32_t id = idesc_bf16(128, 128, false, false);
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
        RowTopk<KCAP> tk;
        tk.init();
        bool ok = true;
        int chunk = 0;
        for (int c0 = 0; c0 < ntile; c0 += kAcc, ++chunk) {
            const int nj = min(kAcc, ntile - c0);
            if (!wait(&sb.acc_full, full_par(chunk))) { ok = false; break; }
            tc_fence_after();
            for (int j = 0; j < nj; ++j) {
                const int kap0 = (c0 + j) * kRows + 32 * cq;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tmem + lane_base + j * 128 + 32 * cq + 16 * q, v);
                    tmem_wait_ld();
                    const int k16 = kap0 + 16 * q;
                    // the candidates of these 16 columns that beat this thread's current
                    // k-th key, then one insertion per warp iteration in lock step
                    float kvs[16];
                    unsigned pend = 0;
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int kap = k16 + u;
                        const float sc = __uint_as_float(v[u]);
                        kvs[u] = (NOISY && kap < lim) ? __fadd_rn(__fmul_rn(sc, sscale), __ldg(nrow + kap)) : sc;
                        if (kap < lim && (!tk.full || kvs[u] > tk.thr)) pend |= 1u << u;
                    }
                    while (__any_sync(0xffffffffu, pend != 0u)) {
                        float ck = -INFINITY, cs = 0.f;     // a lane with nothing pending inserts a no-op
                        int ci = 0x7fffffff;
                        if (pend) {
                            const int u0 = __ffs(pend) - 1;
                            pend &= pend - 1u;
#pragma unroll
                            for (int u = 0; u < 16; ++u)
                                if (u == u0) { ck = kvs[u]; cs = __uint_as_float(v[u]); }
                            ci = k16 + u0;
                        }
                        tk.insert(topk, ck, cs, ci);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sb.acc_empty);
        }
        // merge the four lists of each row through the stage memory (every product
        // that read it has completed: the last accumulators were full)
        float* lk = reinterpret_cast<float*>(sm);                 // [128 rows][4][KCAP] keys
        float* ls = lk + kRows * 4 * KCAP;                         // clean scores
        int* li = reinterpret_cast<int*>(ls + kRows * 4 * KCAP);   // chunks
        const int base = (r * 4 + cq) * KCAP;
#pragma unroll
        for (int p = 0; p < KCAP; ++p) { lk[base + p] = tk.key[p]; ls[base + p] = tk.s[p]; li[base + p] = tk.i[p]; }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpi) : "memory");
        if (cq == 0 && ok && t + 1 <= nC - 1) {
            // four sorted lists of disjoint candidates (entries past a list's end are
            // -inf / no chunk): take the best head k times
            int h[4] = {0, 0, 0, 0};
            const int rb = r * 4 * KCAP;
            RowTopk<KCAP> mg;
            mg.init();
#pragma unroll
            for (int j = 0; j < KCAP; ++j) {
                if (j < topk) {
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
                    mg.key[j] = bk;
                    mg.s[j] = bs;
                    mg.i[j] = bi;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) h[qq] += (best == qq) ? 1 : 0;
                }
            }
            const size_t o = ((size_t)b * nC + t + 1) * topk;
            const int m = lim < topk ? lim : topk;
            float rr[KCAP];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < KCAP; ++j) {
                rr[j] = (j < m) ? mg.s[j] * sscale : -INFINITY;
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
                    idx[o + j] = v ? mg.i[j] : -1;
                    score[o + j] = v ? rr[j] : 0.f;
                    weight[o + j] = v ? expf(rr[j] - mx) / den : 0.f;
                }
            }
        }
        if (R == 0 && r == 0 && cq == 0) {
            // query chunk 0 has no earlier chunk to retrieve
            const size_t o = (size_t)b * nC * topk;
            for (int j = 0; j < topk; ++j) { idx[o + j] = -1; score[o + j] = 0.f; weight[o + j] = 0.f; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int KCAP, bool NOISY>
cudaError_t launch_k(const Shape& sp, const CUtensorMap& tl, const float* noise, int32_t* idx,
                     float* score, float* weight, int* status, cudaStream_t st) {
    auto kern = score_topk_tc_kernel<KCAP, NOISY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((sp.nQ + kRows - 1) / kRows, sp.B);
    GCA_LAUNCH(NOISY ? "score_topk_noisy" : "score_topk", st,
               kern<<<grid, kThreads, kSmem, st>>>(tl, noise, sp.nQ, sp.D, sp.topk, sp.include_self,
                                                  sp.off_by_one, sp.score_scale, idx, score, weight,
                                                  status));
    return cudaGetLastError();
}

}  // namespace

// k <= 16 (the four lists per row live in registers; larger k runs the SIMT
// scorer).  One CTA per 128-row tile takes about the same time however many
// tiles there are (the per-row selection paces it), while the SIMT scorer's
// time grows with the rows, so this path is taken from 16 tiles on (where it
// measured faster: 0.064 against 0.077 ms at 8 x 256 chunks x 768).
bool score_topk_tc_supported(const Shape& sp) {
    const int tiles = sp.B * ((sp.nQ + kRows - 1) / kRows);
    return sp.dtype == GCA_BF16 && sp.D % kBlk == 0 && sp.D <= 8192 && sp.nQ >= 2 && sp.topk <= 16 &&
           tiles >= 16;
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
