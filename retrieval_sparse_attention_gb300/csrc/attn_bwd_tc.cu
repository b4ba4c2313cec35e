// attn_bwd_tc.cu -- GCA backward on the Blackwell tensor cores (bf16, head
// dimension d = 32, 64 or 128).
//
// App. B backward (gradients for Q, K, V and the weights) of the forward
// O_t = sum_j w_j softmax(s q_t K_j^T) V_j.  With p = exp(s q.k - lse_j),
// G_ts = dO_t . v_s and delta_t^j = sum_s p_ts G_ts (= dO_t . O_t^j):
//   dA_ts = w_j p_ts (G_ts - delta_t^j) s,   dQ_t = sum_j sum_s dA_ts k_s,
//   dK_s  = sum over (query chunk, slot) retrieving the chunk of sum_t dA_ts q_t,
//   dV_s  = same of sum_t w_j p_ts dO_t,     dw_j = sum_{t, h} delta_t^j.
//
// Two passes, neither with atomics (every output element is written by
// exactly one CTA, reductions run in a fixed order):
//   pass A, query-major, item = (batch row, query chunk, head): gathers the
//     retrieved chunks' K/V tiles like the forward, recomputes S = Q K^T and
//     G = dO V^T on the tensor cores, forms dA in shared memory and
//     accumulates dQ += dA K in TMEM; it also stores delta and lse per
//     (query chunk, slot, head) as contiguous rows for pass B, and partial dw
//     sums per quarter of the chunk's tokens.
//   pass B, key-major, item = (batch row, pool chunk, head): walks the inverse
//     index of (query chunk, slot) entries that retrieved the chunk, gathers
//     their Q/dO tiles and delta/lse rows, recomputes the scores and dP, and
//     accumulates dK += dA^T Q and dV += (w P)^T dO in TMEM.  For S = 64 a
//     group is a pair of entries whose tiles are stacked into M = 128 products
//     (gca_bwd_kv_pair_kernel); for S = 128 a group is one entry
//     (S^T = K Q^T, G^T = V dO^T, already M = 128).
// Warp roles: warp 0 producer (the whole warp fetches the item metadata --
// slot rows, inverse-index entries and weights -- 32 at a time; lane 0 issues
// the TMA / bulk copies; pass A's item lse block rides on the info barrier as a
// TMA transaction); warp 1 issues the score products into a ring of TMEM
// buffers and owns TMEM (in pass A and the S = 64 pass B the G products come
// from warp 11, a second issuing thread); warp 2 issues the accumulation
// products (dQ, or dK and dV), so neither kind of product waits behind the
// other's issue; warps 3-10 are math warpgroups (two, one for the S = 128
// key-major pass) taking alternate groups and alternate item epilogues; the
// S = 64 math runs on column pairs in packed f32x2 arithmetic.
// Head tiles of d = 64 and 128 are 64-column sub-tiles (128-byte swizzle), of
// d = 32 one 32-column tile (64-byte swizzle); products contract over every
// sub-tile and products with N = d issue one product per sub-tile.  Stage
// counts, item buffers and the number of dK/dV accumulators are chosen per
// (S, d) to fit shared memory and the 512 TMEM columns; at d = 64 and 128 the S = 64
// key-major pass shares one operand pair between its math warpgroups.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace gca {
namespace {

using namespace tc;
using tcx::fast_exp2;
using tcx::kLog2e;
using tcx::pack8;
using tcx::pack8u;
using tcx::Ring;
using tcx::sw128_off;

constexpr int kThreads = 352;         // producer, 2 MMA issuers, 2 math warpgroups
constexpr int kThreadsA = 384;        // + warp 11, which issues the G products (pass A, S = 64 pass B)
constexpr int kInfo = 4;

struct BwdArgs {
    const int32_t* idx;
    const float* w;
    const float* lse;          // [B, Lq, H, topk]
    float* lse2_rows;          // [B, nQ, topk, H, S]: lse * log2(e)
    float* delta_rows;         // [B, nQ, topk, H, S]
    float* dwpart;             // [B, nQ, H, 4, topk]: per TMEM lane quadrant
    const int* offset;         // [B, nP + 1]
    const int* entry;          // [B, nQ * topk]
    const float* entry_w;      // [B, nQ * topk]: the weight of each entry
    const int* order;          // [B, nP]: each row's chunks by descending retrieval count
    int ordered;               // S = 64 key-major pass: deal the items by `order` (else by stride)
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int* status;
    int B, nQ, nP, H, topk, Lq;
    float scale_log2;          // attn_scale * log2(e)
    float attn_scale;
    int n_items;
    int lse_smem;              // pass A: lse blocks staged by TMA (else read per slot)
};

__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

template <int S>
__device__ __forceinline__ void issue_cols16(uint32_t taddr, uint32_t (&r)[16]) {
    if (S == 64) tmem_ld_16x32bx2_x16<64>(taddr, r);
    else tmem_ld_32x32b_x16(taddr, r);
}

template <int S>
__device__ __forceinline__ void load_cols64(uint32_t taddr, float* x) {
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
        uint32_t r[16];
        if (S == 64) tmem_ld_16x32bx2_x16<64>(taddr + 16 * ci, r);
        else tmem_ld_32x32b_x16(taddr + 16 * ci, r);
#pragma unroll
        for (int t = 0; t < 16; ++t) x[16 * ci + t] = __uint_as_float(r[t]);
    }
    tmem_wait_ld();
}

// ============================================================================ pass A
struct ItemInfoA {
    int b, c, h, n;
    int js[kMaxTopk];
    int kaps[kMaxTopk];
    float w[kMaxTopk];
    int8_t code[kMaxTopk];     // 0 valid, otherwise an empty or out-of-range slot
};

template <int S, int DH>
struct CfgA {
    using G = tcx::HeadGeom<DH>;
    static constexpr int M = S;
    static constexpr int NG = S;                           // keys per group
    static constexpr int NSB = (S == 64) ? (DH == 128 ? 2 : 3) : 1;   // S/G TMEM buffers
    // S = 64: dA goes over the S columns of its S/G buffer as the M = 64 A operand of
    // dQ += dA K (row r at lane r % 16 + 32 (r / 16), the layout of the score rows), so
    // the buffer is released by the dQ product, not by the math warps' loads
    static constexpr bool TA = (S == 64);
    // K/V ring depth and Q/dO buffers: what fits beside the P and lse buffers
    static constexpr int STAGES = (S == 64) ? (DH == 128 ? 3 : 8) : (DH == 32 ? 4 : (DH == 64 ? 2 : 1));
    static constexpr int IBUF = (S == 128 && DH == 128) ? 1 : 2;
    static constexpr int TILE = G::tile_bytes(S);
    static constexpr int ITEM_BYTES = 2 * TILE;            // Q then dO
    static constexpr int STAGE_BYTES = 2 * TILE;           // K then V of one slot
    static constexpr int P_BLOCK = M * 128;
    static constexpr int P_BYTES = M * NG * 2;
    static constexpr int OFF_IT = 0;
    static constexpr int OFF_KV = IBUF * ITEM_BYTES;
    static constexpr int OFF_P = OFF_KV + STAGES * STAGE_BYTES;
    // per info-ring entry: the item's lse block, S rows of topk floats
    static constexpr int LSE_TOPK_MAX = (S == 64) ? 16 : 8;
    static constexpr int LSE_BYTES = S * LSE_TOPK_MAX * 4;
    static constexpr int OFF_LSE = OFF_P + 2 * P_BYTES;
    static constexpr int SMEM = OFF_LSE + kInfo * LSE_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t SGW = 2 * S;                 // columns of one S/G buffer
    static constexpr uint32_t COL_DQ = NSB * SGW;          // two dQ accumulators of DH columns
    static_assert(COL_DQ + 2 * DH <= TMEM_COLS, "tensor memory");
    static_assert(STAGES <= 8, "barrier arrays");
    // S/G-full barrier of group qq and the parity of its phase.  With one
    // buffer the two warpgroups alternate on it, so each has its own barrier
    // (kg = the warpgroup's group count).  With several buffers the issuer may
    // run two groups of one warpgroup ahead, so the barrier is per buffer: its
    // next commit needs the buffer's s_empty, i.e. the previous consumer saw it.
    __device__ static int sfull_index(int qq) { return NSB == 1 ? (qq & 1) : qq % NSB; }
    __device__ static uint32_t sfull_par(int qq, int kg) {
        return static_cast<uint32_t>(NSB == 1 ? kg : qq / NSB) & 1u;
    }
};

struct __align__(8) BarsA {
    uint64_t info_full[kInfo], info_empty[kInfo];
    uint64_t it_full[2], it_empty[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[3], s_empty[3];    // per S/G buffer (per warpgroup when one buffer)
    uint64_t p_full[4], p_empty[2];      // p_full: [wg] (S = 128), [group & 3] (S = 64)
    uint64_t o_full[2], o_empty[2];
    uint64_t done, done2, done3;
    uint32_t tmem;
    int abort;
    ItemInfoA info[kInfo];
};

template <int S, int DH>
__global__ void __launch_bounds__(kThreadsA, 1)
gca_bwd_q_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tl, const BwdArgs a) {
    using C = CfgA<S, DH>;
    using HG = tcx::HeadGeom<DH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ BarsA sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kInfo; ++i) {
            mbar_init(&sb.info_full[i], 1);
            mbar_init(&sb.info_empty[i], 3 + 256);     // three MMA issuers + math threads
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.it_full[i], 1);
            mbar_init(&sb.it_empty[i], 2);            // Q read by the S products, dO by the G products
            mbar_init(&sb.p_empty[i], 1);
            mbar_init(&sb.o_full[i], 1);
            mbar_init(&sb.o_empty[i], 128);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&sb.p_full[i], 128);
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&sb.kv_full[i], 1);
            mbar_init(&sb.kv_empty[i], 1);
        }
        for (int i = 0; i < 3; ++i) mbar_init(&sb.s_full[i], 2);   // S issuer + G issuer
        for (int i = 0; i < C::NSB; ++i) mbar_init(&sb.s_empty[i], C::TA ? 1 : 128);
        mbar_init(&sb.done, 1);
        mbar_init(&sb.done2, 1);
        mbar_init(&sb.done3, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tdo);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        if (a.lse_smem) prefetch_tmap(&tl);
    }
    if (warp == 1) {
        tmem_alloc(&sb.tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    if (warp == 0) {
        // The whole warp reads an item's retrieval row (one slot per lane) and
        // compacts its valid slots with a ballot; lane 0 alone waits on
        // barriers and issues the copies.  The item's lse block [S x topk]
        // rides on the info barrier as a TMA transaction.
        constexpr unsigned kAll = 0xffffffffu;
        Ring kv{0, 0}, it{0, 0}, inf{0, 0};
        bool kv_out[C::STAGES] = {}, it_out[2] = {false, false}, inf_out[kInfo] = {};
        uint32_t kv_ph[C::STAGES] = {}, it_ph[2] = {0, 0}, inf_ph[kInfo] = {};
        auto lane0_wait = [&](uint64_t* bar, uint32_t par) {
            int r = 0;
            if (lane == 0) r = wait(bar, par) ? 1 : 0;
            return __shfl_sync(kAll, r, 0) != 0;
        };
        for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
            const int h = item % a.H, bc = item / a.H, c = bc % a.nQ, b = bc / a.nQ;
            const int32_t* row = a.idx + ((size_t)b * a.nQ + c) * a.topk;
            const float* wrow = a.w + ((size_t)b * a.nQ + c) * a.topk;
            int kap0 = -1, kap1 = -1;
            float w0 = 0.f, w1 = 0.f;
            if (lane < a.topk) { kap0 = row[lane]; w0 = wrow[lane]; }
            if (32 + lane < a.topk) { kap1 = row[32 + lane]; w1 = wrow[32 + lane]; }
            if (!lane0_wait(&sb.info_empty[inf.i], inf.ph ^ 1u)) break;
            ItemInfoA& I = sb.info[inf.i];
            int n = 0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int j = 32 * half + lane;
                const int kap = half ? kap1 : kap0;
                const bool okj = j < a.topk && kap >= 0 && kap < a.nP;
                if (j < a.topk) I.code[j] = okj ? 0 : 1;
                const unsigned m = __ballot_sync(kAll, okj);
                if (okj) {
                    const int pos = n + __popc(m & ((1u << lane) - 1u));
                    I.js[pos] = j;
                    I.kaps[pos] = kap;
                    I.w[pos] = half ? w1 : w0;
                }
                n += __popc(m);
            }
            __syncwarp();
            if (lane == 0) {
                I.b = b; I.c = c; I.h = h; I.n = n;
                if (a.lse_smem) {
                    mbar_arrive_expect_tx(&sb.info_full[inf.i], S * a.topk * 4);
                    tma_load_2d(sm + C::OFF_LSE + inf.i * C::LSE_BYTES, &tl, &sb.info_full[inf.i],
                                h * a.topk, b * a.Lq + c * S);
                    inf_out[inf.i] = true;
                    inf_ph[inf.i] = inf.ph;
                } else {
                    mbar_arrive(&sb.info_full[inf.i]);
                }
            }
            inf.next(kInfo);
            if (n == 0) continue;
            if (!lane0_wait(&sb.it_empty[it.i], it.ph ^ 1u)) break;
            if (lane == 0) {
                uint8_t* ib = sm + C::OFF_IT + it.i * C::ITEM_BYTES;
                mbar_arrive_expect_tx(&sb.it_full[it.i], C::ITEM_BYTES);
                for (int sub = 0; sub < HG::SUB; ++sub) {
                    const int off = sub * S * HG::ROW_BYTES;
                    tma_load_2d(ib + off, &tq, &sb.it_full[it.i], h * DH + sub * 64, b * a.Lq + c * S);
                    tma_load_2d(ib + C::TILE + off, &tdo, &sb.it_full[it.i], h * DH + sub * 64,
                                b * a.Lq + c * S);
                }
            }
            it_out[it.i] = true;
            it_ph[it.i] = it.ph;
            it.next(C::IBUF);
            bool ok = true;
            for (int g = 0; g < n; ++g) {
                if (!lane0_wait(&sb.kv_empty[kv.i], kv.ph ^ 1u)) { ok = false; break; }
                if (lane == 0) {
                    uint8_t* stg = sm + C::OFF_KV + kv.i * C::STAGE_BYTES;
                    const int y = (b * a.nP + I.kaps[g]) * S;
                    mbar_arrive_expect_tx(&sb.kv_full[kv.i], 2 * C::TILE);
                    for (int sub = 0; sub < HG::SUB; ++sub) {
                        const int off = sub * S * HG::ROW_BYTES;
                        tma_load_2d(stg + off, &tk, &sb.kv_full[kv.i], h * DH + sub * 64, y);
                        tma_load_2d(stg + C::TILE + off, &tv, &sb.kv_full[kv.i], h * DH + sub * 64, y);
                    }
                }
                kv_out[kv.i] = true;
                kv_ph[kv.i] = kv.ph;
                kv.next(C::STAGES);
            }
            if (!ok) break;
        }
        if (lane == 0) {
            for (int i = 0; i < C::STAGES; ++i)
                if (kv_out[i]) mbar_wait(&sb.kv_full[i], kv_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < C::IBUF; ++i)
                if (it_out[i]) mbar_wait(&sb.it_full[i], it_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < kInfo; ++i)
                if (inf_out[i]) mbar_wait(&sb.info_full[i], inf_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1 || warp == 11) {
        // warp 1: S = Q K^T, warp 11: G = dO V^T of each group (two issuing
        // threads: M = 64 products issue faster from two than from one)
        const bool gs = warp == 11;
        if (lane == 0) {
            Ring kv{0, 0}, it{0, 0}, inf{0, 0};
            int q = 0;
            bool issued = false;
            const uint32_t id_s = idesc_bf16(C::M, S, false, false);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                if (!wait(&sb.info_full[inf.i], inf.ph)) break;
                const int n = sb.info[inf.i].n;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (n == 0) continue;
                if (!wait(&sb.it_full[it.i], it.ph)) break;
                tc_fence_after();
                const uint32_t qaddr = smem_u32(sm + C::OFF_IT + it.i * C::ITEM_BYTES);
                const uint32_t doaddr = qaddr + C::TILE;
                bool ok = true;
                for (int g = 0; g < n; ++g) {
                    const int qq = q + g;
                    const int sbuf = qq % C::NSB;
                    if (!wait(&sb.kv_full[kv.i], kv.ph) ||
                        !wait(&sb.s_empty[sbuf], empty_par(qq / C::NSB))) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(sm + C::OFF_KV + kv.i * C::STAGE_BYTES);
                    const uint32_t vaddr = kaddr + C::TILE;
                    if (gs) tcx::mma_kmajor_dh<DH>(tmem + sbuf * C::SGW + S, doaddr, S, vaddr, S, id_s, 0);
                    else tcx::mma_kmajor_dh<DH>(tmem + sbuf * C::SGW, qaddr, S, kaddr, S, id_s, 0);
                    mma_commit(&sb.s_full[C::sfull_index(qq)]);
                    issued = true;
                    kv.next(C::STAGES);
                }
                if (!ok) break;
                mma_commit(&sb.it_empty[it.i]);     // Q (dO) is read only by these products
                it.next(C::IBUF);
                q += n;
            }
            if (issued) {
                uint64_t* dn = gs ? &sb.done3 : &sb.done;
                mma_commit(dn);
                mbar_wait(dn, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2) {
        // accumulation products: dQ += dA K of each group
        if (lane == 0) {
            Ring kv{0, 0}, inf{0, 0};
            int q = 0, e = 0;
            bool issued = false;
            const uint32_t id_dq = idesc_bf16(C::M, HG::SUB_COLS, false, true);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                if (!wait(&sb.info_full[inf.i], inf.ph)) break;
                const int n = sb.info[inf.i].n;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (n == 0) continue;
                const int ob = e & 1;
                if (!wait(&sb.o_empty[ob], empty_par(e >> 1))) break;
                tc_fence_after();
                const uint32_t d_dq = tmem + C::COL_DQ + ob * DH;
                bool ok = true;
                for (int g = 0; g < n; ++g) {
                    const int qq = q + g, pb = qq & 1;
                    // S = 64: a warpgroup alternates two full barriers (no operand-buffer wait
                    // holds a fast warp back, so its arrival for the next group must not
                    // count toward this one)
                    const bool pf = C::TA ? wait(&sb.p_full[qq & 3], full_par(qq >> 2))
                                          : wait(&sb.p_full[pb], full_par(qq >> 1));
                    if (!pf) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(sm + C::OFF_KV + kv.i * C::STAGE_BYTES);
                    if constexpr (C::TA) {
                        const int sbuf = qq % C::NSB;
                        tcx::mma_ts_mn_dh<DH, S / 16>(d_dq, tmem + sbuf * C::SGW, kaddr, S, id_dq, g > 0);
                        mma_commit(&sb.kv_empty[kv.i]);
                        mma_commit(&sb.s_empty[sbuf]);   // dA (over S) read: the S/G buffer is free
                    } else {
                        const uint32_t paddr = smem_u32(sm + C::OFF_P + pb * C::P_BYTES);
                        tcx::mma_kmajor_mn_dh<DH, S / 16>(d_dq, paddr, C::P_BLOCK, kaddr, S, id_dq, g > 0);
                        // the S / G products of this group are complete (their P exists)
                        mma_commit(&sb.kv_empty[kv.i]);
                        mma_commit(&sb.p_empty[pb]);
                    }
                    issued = true;
                    kv.next(C::STAGES);
                }
                if (!ok) break;
                mma_commit(&sb.o_full[ob]);
                q += n;
                ++e;
            }
            if (issued) {
                mma_commit(&sb.done2);
                mbar_wait(&sb.done2, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp < 11) {
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const int row = (S == 64) ? 16 * qd + (lane & 15) : 32 * qd + lane;
        const int u = (S == 64) ? (lane >> 4) : 0;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        Ring inf{0, 0};
        int q = 0, e = 0, n_all = 0, kg = 0, ko = 0;
        for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++n_all) {
            if (!wait(&sb.info_full[inf.i], inf.ph)) break;
            const ItemInfoA& I = sb.info[inf.i];
            const int b = I.b, c = I.c, h = I.h, n = I.n;
            const size_t tok = (size_t)b * a.Lq + (size_t)c * S + row;
            __nv_bfloat16* dqrow = a.dq + (tok * a.H + h) * DH;
            const bool my_epi = (n == 0) ? ((n_all & 1) == wg) : ((e & 1) == wg);
            float* dwp = a.dwpart + (((size_t)b * a.nQ + c) * a.H + h) * 4 * a.topk;
            if (my_epi && threadIdx.x == 96 + wg * 128)
                for (int j = 0; j < a.topk; ++j)
                    if (I.code[j] != 0)
                        for (int q4 = 0; q4 < 4; ++q4) dwp[q4 * a.topk + j] = 0.f;
            if (n == 0) {
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (my_epi) tcx::zero_acc_row<S, DH>(dqrow, u);
                continue;
            }
            const float* lse_s = reinterpret_cast<const float*>(sm + C::OFF_LSE + inf.i * C::LSE_BYTES);
            bool ok = true;
            for (int g = 0; g < n; ++g) {
                const int qq = q + g;
                if ((qq & 1) != wg) continue;
                const int j = I.js[g];
                const float L2 = (a.lse_smem ? lse_s[row * a.topk + j]
                                             : __ldg(a.lse + (tok * a.H + h) * a.topk + j)) * kLog2e;
                const float wsc = I.w[g] * a.attn_scale;
                const int sbuf = qq % C::NSB;
                if (!wait(&sb.s_full[C::sfull_index(qq)], C::sfull_par(qq, kg))) { ok = false; break; }
                tc_fence_after();
                const uint32_t ts0 = tmem + lane_base + sbuf * C::SGW;
                const uint32_t tg0 = ts0 + S;
                uint8_t* pb = sm + C::OFF_P + wg * C::P_BYTES;
                float dl = 0.f;
                // the row's delta and lse*log2(e) for the key-major pass, and this
                // warp's partial of dw (for S = 64 both halves of the warp hold the
                // same rows' delta: reduce within one); for S = 64 issued before
                // the P buffer wait so the stores overlap it
                auto emit_rows = [&](float dlv) {
                    if (u == 0) {
                        const size_t rr = ((((size_t)b * a.nQ + c) * a.topk + j) * a.H + h) * S + row;
                        a.delta_rows[rr] = dlv;
                        a.lse2_rows[rr] = L2;
                    }
                    float part = dlv;
#pragma unroll
                    for (int o2 = (S == 64 ? 8 : 16); o2 > 0; o2 >>= 1)
                        part += __shfl_xor_sync(0xffffffffu, part, o2);
                    if (lane == 0) dwp[qd * a.topk + j] = part;
                };
                if constexpr (S == 64) {
                    // this thread: one token row, keys u*32 .. u*32+31 of the slot
                    uint32_t r0[16], r1[16], r2[16], r3[16];
                    tmem_ld_16x32bx2_x16<32>(ts0, r0);
                    tmem_ld_16x32bx2_x16<32>(ts0 + 16, r1);
                    tmem_ld_16x32bx2_x16<32>(tg0, r2);
                    tmem_ld_16x32bx2_x16<32>(tg0 + 16, r3);
                    tmem_wait_ld();
                    // column pairs in packed f32x2 arithmetic: p = exp2(s sl - L2) as
                    // exp2(-(L2 - s sl)), delta = sum p g, dA = p (g - delta) w scale
                    const uint64_t nsl2 = tcx::f2_pack(-a.scale_log2, -a.scale_log2);
                    const uint64_t l2_2 = tcx::f2_pack(L2, L2);
                    uint64_t pr2[16], gv2[16];
                    uint64_t dacc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        const uint32_t* rs = p < 8 ? r0 : r1;
                        const uint32_t* rg = p < 8 ? r2 : r3;
                        const int t = 2 * (p & 7);
                        float y0, y1;
                        tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(__uint_as_float(rs[t]), __uint_as_float(rs[t + 1])),
                                                  nsl2, l2_2), y0, y1);
                        pr2[p] = tcx::f2_pack(fast_exp2(-y0), fast_exp2(-y1));
                        gv2[p] = tcx::f2_pack(__uint_as_float(rg[t]), __uint_as_float(rg[t + 1]));
                        dacc[p & 3] = tcx::ffma2(pr2[p], gv2[p], dacc[p & 3]);
                    }
                    float d8[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) tcx::f2_unpack(dacc[i], d8[2 * i], d8[2 * i + 1]);
                    dl = ((d8[0] + d8[1]) + (d8[2] + d8[3])) + ((d8[4] + d8[5]) + (d8[6] + d8[7]));
                    dl += __shfl_xor_sync(0xffffffffu, dl, 16);     // the row's other 32 keys
                    emit_rows(dl);
                    const uint64_t wsc2 = tcx::f2_pack(wsc, wsc), ndl2 = tcx::f2_pack(-dl * wsc, -dl * wsc);
                    uint32_t pk[16];
#pragma unroll
                    for (int p = 0; p < 16; ++p)
                        pk[p] = tcx::pack_bf16x2(tcx::fmul2(pr2[p], tcx::ffma2(gv2[p], wsc2, ndl2)));
                    // dA over the S columns 16 u .. 16 u + 15 of this row (keys 32 u ..): the
                    // warp's loads have completed, so the scores there are in registers
                    tmem_st_16x32bx2_x16<16>(ts0, pk);
                    tmem_wait_st();
                } else {
                    // this thread: one token row, all 128 keys in two 64-key chunks
                    float x[64];
                    for (int ch = 0; ch < 2; ++ch) {
                        load_cols64<S>(ts0 + ch * 64, x);
#pragma unroll
                        for (int i = 0; i < 64; ++i) x[i] = fast_exp2(fmaf(x[i], a.scale_log2, -L2));
                        float d8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) d8[i] = 0.f;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t g0[16], g1[16];
                            issue_cols16<S>(tg0 + ch * 64 + 32 * half, g0);
                            issue_cols16<S>(tg0 + ch * 64 + 32 * half + 16, g1);
                            tmem_wait_ld();
#pragma unroll
                            for (int t = 0; t < 16; ++t) {
                                d8[t & 7] = fmaf(x[32 * half + t], __uint_as_float(g0[t]), d8[t & 7]);
                                d8[t & 7] = fmaf(x[32 * half + 16 + t], __uint_as_float(g1[t]), d8[t & 7]);
                            }
                        }
                        dl += ((d8[0] + d8[1]) + (d8[2] + d8[3])) + ((d8[4] + d8[5]) + (d8[6] + d8[7]));
                    }
                    if (!wait(&sb.p_empty[wg], empty_par(kg))) { ok = false; break; }
                    for (int ch = 0; ch < 2; ++ch) {
                        load_cols64<S>(ts0 + ch * 64, x);
#pragma unroll
                        for (int i = 0; i < 64; ++i) x[i] = fast_exp2(fmaf(x[i], a.scale_log2, -L2));
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t g0[16], g1[16];
                            issue_cols16<S>(tg0 + ch * 64 + 32 * half, g0);
                            issue_cols16<S>(tg0 + ch * 64 + 32 * half + 16, g1);
                            tmem_wait_ld();
                            if (ch == 1 && half == 1) {
                                tc_fence_before();
                                mbar_arrive(&sb.s_empty[sbuf]);
                            }
                            float gg[32];
#pragma unroll
                            for (int t = 0; t < 16; ++t) {
                                gg[t] = x[32 * half + t] * (__uint_as_float(g0[t]) - dl);
                                gg[16 + t] = x[32 * half + 16 + t] * (__uint_as_float(g1[t]) - dl);
                            }
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4)
                                *reinterpret_cast<uint4*>(pb + ch * C::P_BLOCK + sw128_off(row, 4 * half + c4)) =
                                    pack8(gg + 8 * c4, wsc);
                        }
                    }
                }
                if constexpr (C::TA) {
                    tc_fence_before();
                    mbar_arrive(&sb.p_full[qq & 3]);
                } else {
                    fence_proxy_async_smem();
                    mbar_arrive(&sb.p_full[wg]);
                }
                ++kg;
                if constexpr (S != 64) emit_rows(dl);     // (S = 64 emitted them before the P wait)
            }
            mbar_arrive(&sb.info_empty[inf.i]);
            inf.next(kInfo);
            if (!ok) break;
            q += n;
            const bool mine = (e & 1) == wg;
            ++e;
            if (!mine) continue;
            if (!wait(&sb.o_full[wg], full_par(ko))) break;
            ++ko;
            tc_fence_after();
            tcx::store_acc_row<S, DH>(tmem + lane_base + C::COL_DQ + wg * DH, dqrow, u);
            tc_fence_before();
            mbar_arrive(&sb.o_empty[wg]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, CfgA<S, DH>::TMEM_COLS);
    }
}

// ============================================================================ pass B
struct ItemInfoB {
    int b, kap, h, ne;
};

struct EntryInfo {
    int c, j;
    float w;
    int pad;
};

struct __align__(8) BarsB {
    uint64_t info_full[kInfo], info_empty[kInfo];
    uint64_t it_full[2], it_empty[2];
    uint64_t st_full[6], st_empty[6];
    uint64_t s_full[2], s_empty[2];    // s_full per math warpgroup, s_empty per S/G buffer
    uint64_t p_full[2], p_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t done, done2, done3;
    uint32_t tmem;
    int abort;
    ItemInfoB info[kInfo];
};

// The key-major pass for S = 128 (S = 64 uses the entry-pair kernel below).
// Work unit = (inverse-index entry, half of its 128 query tokens).  Per unit
// S^T = K Q_h^T and G^T = V dO_h^T are M = 128 (keys) x N = 64 (tokens)
// products into a 128-column TMEM half-buffer (S^T, then G^T).  A math thread
// owns one key row: it reads its 64 scores and 64 G values in two pieces of 32
// tokens and writes dA^T (bf16 pairs) over the S^T columns and w P^T over the
// G^T columns it has already read -- the row of key s is TMEM lane s, exactly
// the layout of an A operand -- so dK += dA^T Q_h and dV += (w P)^T dO_h read A
// from tensor memory (K = 64 tokens) and no shared-memory operand buffer
// exists.  Two math warpgroups take alternate units; dK and dV are issued by
// two threads, S^T and G^T by one.
template <int DH>
struct CfgK {
    using G = tcx::HeadGeom<DH>;
    static constexpr int S = 128;
    static constexpr int TILE = G::tile_bytes(S);         // 128 rows x DH
    static constexpr int ITEM_BYTES = 2 * TILE;           // K then V
    static constexpr int IBUF = DH == 128 ? 1 : 2;
    static constexpr int VEC_OFF = 2 * TILE;              // after the Q and dO tiles
    static constexpr int ENT_OFF = VEC_OFF + 1024;        // lse2[128], delta[128], then entry info
    static constexpr int STAGE_BYTES = VEC_OFF + 2048;
    static constexpr int STAGES = DH == 32 ? 6 : (DH == 64 ? 4 : 2);
    static constexpr int OFF_IT = 0;
    static constexpr int OFF_ST = IBUF * ITEM_BYTES;
    static constexpr int SMEM = OFF_ST + STAGES * STAGE_BYTES + 1024;
    static constexpr int NHB = DH == 128 ? 2 : 3;         // TMEM half-buffers of 128 columns
    static constexpr int NACC = DH == 32 ? 2 : 1;         // dK/dV accumulators
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_ACC = NHB * 128;        // dK then dV (DH columns each) per accumulator
    static_assert(COL_ACC + NACC * 2 * DH <= TMEM_COLS, "tensor memory");
    static_assert(STAGES <= 6, "barrier arrays");
};

struct __align__(8) BarsK {
    uint64_t info_full[kInfo], info_empty[kInfo];
    uint64_t it_full[2], it_empty[2];
    uint64_t st_full[6], st_empty[6];
    uint64_t s_full[3], s_empty[3];    // per TMEM half-buffer
    uint64_t p_full[4];                // per unit, cycling four (two per warpgroup)
    uint64_t o_full[2], o_empty[2];    // o_full per storing warpgroup, o_empty per accumulator
    uint64_t done, done2, done3;
    uint32_t tmem;
    int abort;
    ItemInfoB info[kInfo];
};

template <int DH>
__global__ void __launch_bounds__(kThreadsA, 1)
gca_bwd_kv128_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     const BwdArgs a) {
    using C = CfgK<DH>;
    using HG = tcx::HeadGeom<DH>;
    constexpr int S = C::S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ BarsK sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };
    const int nE = a.nQ * a.topk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kInfo; ++i) {
            mbar_init(&sb.info_full[i], 1);
            mbar_init(&sb.info_empty[i], 3 + 256);     // three MMA issuers + math threads
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.it_full[i], 1);
            mbar_init(&sb.it_empty[i], 1);
            mbar_init(&sb.o_full[i], 2);              // the dK issuer + the dV issuer
            mbar_init(&sb.o_empty[i], 128);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&sb.p_full[i], 128);
        for (int i = 0; i < C::NHB; ++i) {
            mbar_init(&sb.s_full[i], 1);
            mbar_init(&sb.s_empty[i], 2);             // freed by the dK and dV products
        }
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&sb.st_full[i], 1);
            mbar_init(&sb.st_empty[i], 2);
        }
        mbar_init(&sb.done, 1);
        mbar_init(&sb.done2, 1);
        mbar_init(&sb.done3, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tdo);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 1) {
        tmem_alloc(&sb.tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    if (warp == 0) {
        // Producer: the whole warp walks the items; lane 0 alone waits on barriers
        // and issues the copies.  The other lanes fetch the item offsets and the
        // entry records (entry, weight) 32 at a time.
        constexpr unsigned kAll = 0xffffffffu;
        Ring st{0, 0}, it{0, 0}, inf{0, 0};
        bool st_out[C::STAGES] = {}, it_out[2] = {false, false};
        uint32_t st_ph[C::STAGES] = {}, it_ph[2] = {0, 0};
        auto lane0_wait = [&](uint64_t* bar, uint32_t par) {
            int r = 0;
            if (lane == 0) r = wait(bar, par) ? 1 : 0;
            return __shfl_sync(kAll, r, 0) != 0;
        };
        int my_e0 = 0, my_ne = 0;
        int n_item = 0;
        for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++n_item) {
            if ((n_item & 31) == 0) {
                const int it_l = item + lane * gridDim.x;
                my_e0 = my_ne = 0;
                if (it_l < a.n_items) {
                    const int bk_l = it_l / a.H, kap_l = bk_l % a.nP, b_l = bk_l / a.nP;
                    const int* off = a.offset + (size_t)b_l * (a.nP + 1) + kap_l;
                    my_e0 = off[0];
                    my_ne = off[1] - my_e0;
                }
            }
            const int e0 = __shfl_sync(kAll, my_e0, n_item & 31);
            const int ne = __shfl_sync(kAll, my_ne, n_item & 31);
            const int h = item % a.H, bk = item / a.H, kap = bk % a.nP, b = bk / a.nP;
            if (!lane0_wait(&sb.info_empty[inf.i], inf.ph ^ 1u)) break;
            if (lane == 0) {
                ItemInfoB& I = sb.info[inf.i];
                I.b = b; I.kap = kap; I.h = h; I.ne = ne;
                mbar_arrive(&sb.info_full[inf.i]);
            }
            inf.next(kInfo);
            if (ne <= 0) continue;
            if (!lane0_wait(&sb.it_empty[it.i], it.ph ^ 1u)) break;
            if (lane == 0) {
                uint8_t* ib = sm + C::OFF_IT + it.i * C::ITEM_BYTES;
                mbar_arrive_expect_tx(&sb.it_full[it.i], C::ITEM_BYTES);
                for (int sub = 0; sub < HG::SUB; ++sub) {
                    const int off = sub * S * HG::ROW_BYTES;
                    tma_load_2d(ib + off, &tk, &sb.it_full[it.i], h * DH + sub * 64, (b * a.nP + kap) * S);
                    tma_load_2d(ib + C::TILE + off, &tv, &sb.it_full[it.i], h * DH + sub * 64,
                                (b * a.nP + kap) * S);
                }
            }
            it_out[it.i] = true;
            it_ph[it.i] = it.ph;
            it.next(C::IBUF);
            bool ok = true;
            for (int base = 0; base < ne && ok; base += 32) {
                int my_c = 0, my_j = 0;
                float my_w = 0.f;
                if (base + lane < ne) {
                    const size_t at = (size_t)b * nE + e0 + base + lane;
                    const int e = a.entry[at];
                    my_c = e / a.topk;
                    my_j = e % a.topk;
                    my_w = a.entry_w[at];
                }
                const int cnt = min(32, ne - base);
                for (int u = 0; u < cnt; ++u) {
                    const int c = __shfl_sync(kAll, my_c, u);
                    const int j = __shfl_sync(kAll, my_j, u);
                    const float wv = __shfl_sync(kAll, my_w, u);
                    if (!lane0_wait(&sb.st_empty[st.i], st.ph ^ 1u)) { ok = false; break; }
                    if (lane == 0) {
                        uint8_t* stg = sm + C::OFF_ST + st.i * C::STAGE_BYTES;
                        EntryInfo* ei = reinterpret_cast<EntryInfo*>(stg + C::ENT_OFF);
                        ei->c = c; ei->j = j; ei->w = wv;
                        mbar_arrive_expect_tx(&sb.st_full[st.i], 2 * C::TILE + 2 * S * 4);
                        for (int sub = 0; sub < HG::SUB; ++sub) {
                            const int off = sub * S * HG::ROW_BYTES;
                            tma_load_2d(stg + off, &tq, &sb.st_full[st.i], h * DH + sub * 64, b * a.Lq + c * S);
                            tma_load_2d(stg + C::TILE + off, &tdo, &sb.st_full[st.i], h * DH + sub * 64,
                                        b * a.Lq + c * S);
                        }
                        const size_t rb = ((((size_t)b * a.nQ + c) * a.topk + j) * a.H + h) * S;
                        tcx::bulk_load(stg + C::VEC_OFF, a.lse2_rows + rb, S * 4, &sb.st_full[st.i]);
                        tcx::bulk_load(stg + C::VEC_OFF + S * 4, a.delta_rows + rb, S * 4, &sb.st_full[st.i]);
                    }
                    st_out[st.i] = true;
                    st_ph[st.i] = st.ph;
                    st.next(C::STAGES);
                }
            }
            if (!ok) break;
        }
        if (lane == 0) {
            for (int i = 0; i < C::STAGES; ++i)
                if (st_out[i]) mbar_wait(&sb.st_full[i], st_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < C::IBUF; ++i)
                if (it_out[i]) mbar_wait(&sb.it_full[i], it_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // S^T = K Q_h^T and G^T = V dO_h^T of each unit (M = 128 keys, N = 64 tokens)
        if (lane == 0) {
            Ring st{0, 0}, it{0, 0}, inf{0, 0};
            int u = 0;                          // units issued
            bool issued = false;
            const uint32_t id_s = idesc_bf16(128, 64, false, false);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                if (!wait(&sb.info_full[inf.i], inf.ph)) break;
                const int ne = sb.info[inf.i].ne;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (ne <= 0) continue;
                if (!wait(&sb.it_full[it.i], it.ph)) break;
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sm + C::OFF_IT + it.i * C::ITEM_BYTES);
                const uint32_t vaddr = kaddr + C::TILE;
                bool ok = true;
                for (int g = 0; g < ne && ok; ++g) {
                    if (!wait(&sb.st_full[st.i], st.ph)) { ok = false; break; }
                    const uint32_t qaddr = smem_u32(sm + C::OFF_ST + st.i * C::STAGE_BYTES);
                    const uint32_t doaddr = qaddr + C::TILE;
                    for (int hf = 0; hf < 2; ++hf, ++u) {
                        const int hb = u % C::NHB;
                        if (!wait(&sb.s_empty[hb], empty_par(u / C::NHB))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t d = tmem + hb * 128;
                        tcx::mma_kmajor_dh<DH>(d, kaddr, S, qaddr + 64 * hf * HG::ROW_BYTES, S, id_s, 0);
                        tcx::mma_kmajor_dh<DH>(d + 64, vaddr, S, doaddr + 64 * hf * HG::ROW_BYTES, S, id_s, 0);
                        mma_commit(&sb.s_full[hb]);
                        issued = true;
                    }
                    st.next(C::STAGES);
                }
                if (!ok) break;
                mma_commit(&sb.it_empty[it.i]);     // K and V are read only by these products
                it.next(C::IBUF);
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2 || warp == 11) {
        // warp 2: dK += dA^T Q_h, warp 11: dV += (w P)^T dO_h, A from TMEM (K = 64 tokens)
        const bool dvi = warp == 11;
        if (lane == 0) {
            Ring st{0, 0}, inf{0, 0};
            int u = 0, e = 0;
            bool issued = false;
            const uint32_t id_acc = idesc_bf16(128, HG::SUB_COLS, false, true);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                if (!wait(&sb.info_full[inf.i], inf.ph)) break;
                const int ne = sb.info[inf.i].ne;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (ne <= 0) continue;
                const int ob = e % C::NACC;
                if (!wait(&sb.o_empty[ob], empty_par(e / C::NACC))) break;
                tc_fence_after();
                const uint32_t d_acc = tmem + C::COL_ACC + ob * 2 * DH + (dvi ? DH : 0);
                bool ok = true;
                for (int g = 0; g < ne && ok; ++g) {
                    const uint32_t stg = smem_u32(sm + C::OFF_ST + st.i * C::STAGE_BYTES);
                    const uint32_t xaddr = stg + (dvi ? C::TILE : 0);    // Q (dK) or dO (dV)
                    for (int hf = 0; hf < 2; ++hf, ++u) {
                        const int hb = u % C::NHB;
                        if (!wait(&sb.p_full[u & 3], full_par(u >> 2))) { ok = false; break; }
                        tc_fence_after();
                        tcx::mma_ts_mn_dh<DH, 4>(d_acc, tmem + hb * 128 + (dvi ? 64 : 0),
                                                 xaddr + 64 * hf * HG::ROW_BYTES, S, id_acc,
                                                 (g > 0 || hf > 0) ? 1u : 0u);
                        mma_commit(&sb.s_empty[hb]);
                        issued = true;
                    }
                    if (!ok) break;
                    mma_commit(&sb.st_empty[st.i]);
                    st.next(C::STAGES);
                }
                if (!ok) break;
                // the full barrier belongs to the warpgroup that stores this item
                mma_commit(&sb.o_full[e & 1]);
                ++e;
            }
            if (issued) {
                uint64_t* dn = dvi ? &sb.done3 : &sb.done2;
                mma_commit(dn);
                mbar_wait(dn, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp < 11) {
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const int row = 32 * qd + lane;             // key row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        Ring inf{0, 0}, st{0, 0};
        int u = 0, e = 0, n_all = 0;
        for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++n_all) {
            if (!wait(&sb.info_full[inf.i], inf.ph)) break;
            const ItemInfoB I = sb.info[inf.i];
            mbar_arrive(&sb.info_empty[inf.i]);
            inf.next(kInfo);
            const size_t krow = (size_t)(I.b * a.nP + I.kap) * S + row;
            __nv_bfloat16* dkrow = a.dk + (krow * a.H + I.h) * DH;
            __nv_bfloat16* dvrow = a.dv + (krow * a.H + I.h) * DH;
            if (I.ne <= 0) {
                if ((n_all & 1) == wg) {
                    tcx::zero_acc_row<128, DH>(dkrow, 0);
                    tcx::zero_acc_row<128, DH>(dvrow, 0);
                }
                continue;
            }
            bool ok = true;
            for (int g = 0; g < I.ne && ok; ++g) {
                const int stage = st.i;
                const uint32_t stph = st.ph;
                st.next(C::STAGES);
                for (int hf = 0; hf < 2; ++hf, ++u) {
                    if ((u & 1) != wg) continue;
                    const int hb = u % C::NHB;
                    // own s_full first: its completion implies this entry's stage has
                    // landed, so the stage barrier's phase below is unambiguous
                    if (!wait(&sb.s_full[hb], full_par(u / C::NHB)) || !wait(&sb.st_full[stage], stph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* stg = sm + C::OFF_ST + stage * C::STAGE_BYTES;
                    const EntryInfo ei = reinterpret_cast<const EntryInfo*>(stg + C::ENT_OFF)[0];
                    const float wv = ei.w, wsc = wv * a.attn_scale;
                    const float* vec = reinterpret_cast<const float*>(stg + C::VEC_OFF) + 64 * hf;
                    const uint32_t tb = tmem + lane_base + hb * 128;
#pragma unroll
                    for (int pc = 0; pc < 2; ++pc) {
                        // tokens 64 hf + 32 pc .. + 31 of this key row
                        uint32_t rx[32], ry[32];
                        tmem_ld_32x32b_x32(tb + 32 * pc, rx);
                        tmem_ld_32x32b_x32(tb + 64 + 32 * pc, ry);
                        tmem_wait_ld();
                        const uint32_t* r0 = rx;
                        const uint32_t* r1 = rx + 16;
                        const uint32_t* r2 = ry;
                        const uint32_t* r3 = ry + 16;
                        uint32_t pa[16], pp[16];
#pragma unroll
                        for (int p2 = 0; p2 < 16; ++p2) {
                            const uint32_t* rs = p2 < 8 ? r0 : r1;
                            const uint32_t* rg = p2 < 8 ? r2 : r3;
                            const int tt = 2 * (p2 & 7);
                            const int t0 = 32 * pc + 2 * p2;
                            const float pr0 = fast_exp2(fmaf(__uint_as_float(rs[tt]), a.scale_log2, -vec[t0]));
                            const float pr1 = fast_exp2(fmaf(__uint_as_float(rs[tt + 1]), a.scale_log2, -vec[t0 + 1]));
                            pa[p2] = tcx::pack_bf16(pr0 * (__uint_as_float(rg[tt]) - vec[128 + t0]) * wsc,
                                                    pr1 * (__uint_as_float(rg[tt + 1]) - vec[128 + t0 + 1]) * wsc);
                            pp[p2] = tcx::pack_bf16(pr0 * wv, pr1 * wv);
                        }
                        // dA^T over S^T columns 16 pc .., w P^T over G^T columns 16 pc .. (both read)
                        tmem_st_32x32b_x16(tb + 16 * pc, pa);
                        tmem_st_32x32b_x16(tb + 64 + 16 * pc, pp);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&sb.p_full[u & 3]);
                }
            }
            if (!ok) break;
            const bool mine = (e & 1) == wg;
            const int ob = e % C::NACC, ko = e >> 1;
            ++e;
            if (!mine) continue;
            if (!wait(&sb.o_full[wg], full_par(ko))) break;
            tc_fence_after();
            const uint32_t acc = tmem + lane_base + C::COL_ACC + ob * 2 * DH;
            tcx::store_acc_row<128, DH>(acc, dkrow, 0);
            tcx::store_acc_row<128, DH>(acc + DH, dvrow, 0);
            tc_fence_before();
            mbar_arrive(&sb.o_empty[ob]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, CfgK<DH>::TMEM_COLS);
    }
}

// ============================================================================ pass B, S = 64
// Item = (row, pool chunk, head) as above; a group is a PAIR of inverse-index
// entries (two query chunks that retrieved this chunk, or one for an odd
// tail).  Their Q tiles (and dO tiles) sit one above the other in the stage, so
// S = [Q_1; Q_2] K^T and G = [dO_1; dO_2] V^T are M = 128 products (full rate,
// all 128 TMEM lanes, four MMAs each per pair instead of eight per entry at
// M = 64).  A math thread owns one query row of the pair: its lse and delta are
// scalars, and it writes its 64 keys of w P and dA as one 128-byte row, which
// the accumulation products read as MN-major A operands:
// dK += dA^T [Q_1; Q_2] and dV += (w P)^T [dO_1; dO_2] over K = 128 queries
// (64 for a single entry).
// The order in which the S = 64 key-major pass deals its items.  An item's cost is
// the number of entry pairs of its chunk, and a fixed stride over items in index
// order leaves the busiest CTA ~5% above the mean.  One CTA per batch row ranks the
// row's chunks by retrieval count (descending, counts above 255 taken as 255; ties by
// chunk index) with a stable counting sort: a histogram of the counts, its scan from
// the top, and each chunk's place among equal counts from warp matches plus the
// per-warp counts of the warps before it.  The dealt sequence takes the rows one after
// another (so the Q / dO in flight is one batch row's, not every row's) and
// snakes: position p is head p % H of rank k = (p / H) % nP of row b = p / (nP H),
// ranks descending in the last row and in every second row before it, ascending in
// the others, so the cost of consecutive positions never jumps at a row boundary.
// Round r of the CTAs takes positions r G .. r G + G - 1 boustrophedon (CTA c takes
// c in even rounds, G - 1 - c in odd ones).
__global__ void __launch_bounds__(1024) pair_order_kernel(const int* __restrict__ count, int nP,
                                                          int* __restrict__ order) {
    __shared__ int hist[256];
    __shared__ int start[256];
    __shared__ int per_warp[32][256];      // chunks of each count in each warp
    const int b = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const bool real = t < nP;
    const int key = real ? min(count[(size_t)b * nP + t], 255) : -1;
    if (t < 256) hist[t] = 0;
    for (int i = t; i < 32 * 256; i += 1024) (&per_warp[0][0])[i] = 0;
    __syncthreads();
    // equal keys in this warp: the lowest such lane records the warp's count of the key
    const unsigned same = __match_any_sync(0xffffffffu, key);
    const int in_warp = __popc(same & ((1u << lane) - 1u));
    if (real) {
        atomicAdd(&hist[key], 1);
        if (in_warp == 0) per_warp[warp][key] = __popc(same);
    }
    __syncthreads();
    if (warp == 0) {                       // start[k] = chunks with a larger count
        int v[8], run = 0;
        for (int i = 0; i < 8; ++i) { v[i] = hist[255 - (8 * lane + i)]; run += v[i]; }
        int incl = run;
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        int acc = incl - run;
        for (int i = 0; i < 8; ++i) { start[255 - (8 * lane + i)] = acc; acc += v[i]; }
    }
    __syncthreads();
    if (real) {
        int pos = start[key] + in_warp;
        for (int w = 0; w < warp; ++w) pos += per_warp[w][key];
        order[(size_t)b * nP + pos] = t;
    }
}

// Position of round r for CTA c (boustrophedon when the items are dealt by rank).
__device__ __forceinline__ int pair_pos(const BwdArgs& a, int r) {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((a.ordered && (r & 1)) ? G - 1 - c : c);
}
// Item at position p: (row b, chunk of rank k in row b, head h), or p itself when not ordered.
__device__ __forceinline__ int pair_item(const BwdArgs& a, int p) {
    if (!a.ordered) return p;
    const int bk = p / a.H, h = p - bk * a.H, b = bk / a.nP;
    int k = bk - b * a.nP;
    if ((a.B - 1 - b) & 1) k = a.nP - 1 - k;     // snake: rows alternate, the last one descends
    return (b * a.nP + a.order[(size_t)b * a.nP + k]) * a.H + h;
}

template <int DH, bool SHARE>
struct CfgP {
    using G = tcx::HeadGeom<DH>;
    static constexpr int S = 64;
    static constexpr int TILE = G::tile_bytes(64);        // 64 rows x DH bf16
    static constexpr int ITEM_BYTES = 2 * TILE;           // K then V
    // what fits: d = 128 keeps one K/V item buffer and one operand pair shared
    // by both math warpgroups, and a single dK/dV accumulator in TMEM; at d = 64
    // (SHARE) a shared operand pair buys a second K/V item buffer, which hides
    // the K/V load at item boundaries: worth more than private pairs when items
    // hold few entries
    static constexpr int STAGES = DH == 32 ? 4 : (DH == 64 ? 4 : 2);
    static constexpr int IBUF = DH == 32 || (DH == 64 && SHARE) ? 2 : 1;
    static constexpr bool SHARED_P = DH == 128 || (DH == 64 && SHARE);
    static constexpr int NACC = DH == 128 ? 1 : 2;
    // Q of entries 0 and 1: sub-tile s holds rows 0-63 (entry 0) then 64-127
    // (entry 1), so [Q_1; Q_2] is one 128-row operand per sub-tile
    static constexpr int Q_OFF = 0;
    static constexpr int DO_OFF = 2 * TILE;               // dO of entries 0 and 1, likewise
    static constexpr int VEC_OFF = 4 * TILE;              // lse2[2][64], then delta[2][64]
    static constexpr int ENT_OFF = VEC_OFF + 1024;        // EntryInfo[2]
    static constexpr int STAGE_BYTES = VEC_OFF + 2048;
    static constexpr int ENTRY_TX = 2 * TILE + 2 * 64 * 4;
    static constexpr int P_BYTES = 128 * 128;             // one operand: 128 query rows x 64 keys
    static constexpr int OFF_IT = 0;
    static constexpr int OFF_ST = IBUF * ITEM_BYTES;
    static constexpr int OFF_P = OFF_ST + STAGES * STAGE_BYTES;
    static constexpr int SMEM = OFF_P + (SHARED_P ? 1 : 2) * 2 * P_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t SGW = 128;                  // S (64 columns), then G
    static constexpr uint32_t COL_ACC = 2 * SGW;          // dK then dV (DH columns each) per buffer
    static_assert(COL_ACC + NACC * 2 * DH <= TMEM_COLS, "tensor memory");
    static_assert(STAGES <= 6, "barrier arrays");
};

template <int DH, bool SHARE>
__global__ void __launch_bounds__(kThreadsA, 1)
gca_bwd_kv_pair_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                       const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const BwdArgs a) {
    using C = CfgP<DH, SHARE>;
    using HG = tcx::HeadGeom<DH>;
    constexpr int S = C::S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ BarsB sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };
    const int nE = a.nQ * a.topk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kInfo; ++i) {
            mbar_init(&sb.info_full[i], 1);
            mbar_init(&sb.info_empty[i], 3 + 256);     // three MMA issuers + math threads
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.it_full[i], 1);
            mbar_init(&sb.it_empty[i], 1);            // K and V read by the S and G products
            mbar_init(&sb.p_full[i], 128);
            mbar_init(&sb.p_empty[i], 2);             // the dK issuer + the dV issuer
            mbar_init(&sb.o_full[i], 2);
            mbar_init(&sb.o_empty[i], 128);
            mbar_init(&sb.s_full[i], 1);
            mbar_init(&sb.s_empty[i], 128);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&sb.st_full[i], 1);
            mbar_init(&sb.st_empty[i], 2);            // Q read by the dK products, dO by the dV products
        }
        mbar_init(&sb.done, 1);
        mbar_init(&sb.done2, 1);
        mbar_init(&sb.done3, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tdo);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 1) {
        tmem_alloc(&sb.tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    if (warp == 0) {
        // Producer: the whole warp walks the items; lane 0 alone waits and issues
        // the copies.  Item offsets are fetched 32 items at a time and entry records
        // (entry, weight) 32 entries at a time, one per lane; the next item's offsets
        // and first records are loaded while this item is staged, so no dependent
        // global load sits between two items.  Entries are staged in pairs.
        constexpr unsigned kAll = 0xffffffffu;
        Ring st{0, 0}, it{0, 0}, inf{0, 0};
        bool st_out[C::STAGES] = {}, it_out[2] = {false, false};
        uint32_t st_ph[C::STAGES] = {}, it_ph[2] = {0, 0};
        auto lane0_wait = [&](uint64_t* bar, uint32_t par) {
            int r = 0;
            if (lane == 0) r = wait(bar, par) ? 1 : 0;
            return __shfl_sync(kAll, r, 0) != 0;
        };
        int my_item = a.n_items, my_e0 = 0, my_ne = 0;   // lane l: item and offsets of round r0 + l
        auto load_offsets = [&](int r0) {
            const int p_l = pair_pos(a, r0 + lane);
            my_item = a.n_items;
            my_e0 = my_ne = 0;
            if (p_l < a.n_items) {
                my_item = pair_item(a, p_l);
                const int bk_l = my_item / a.H, kap_l = bk_l % a.nP, b_l = bk_l / a.nP;
                const int* off = a.offset + (size_t)b_l * (a.nP + 1) + kap_l;
                my_e0 = off[0];
                my_ne = off[1] - my_e0;
            }
        };
        auto fetch = [&](int b_, int e0_, int ne_, int base, int& e_out, float& w_out) {
            e_out = 0;
            w_out = 0.f;
            if (base + lane < ne_) {
                const size_t at = (size_t)b_ * nE + e0_ + base + lane;
                e_out = a.entry[at];
                w_out = a.entry_w[at];
            }
        };
        int n_item = 0;
        load_offsets(0);
        int item = __shfl_sync(kAll, my_item, 0);
        int nx_e0 = __shfl_sync(kAll, my_e0, 0), nx_ne = __shfl_sync(kAll, my_ne, 0);
        int nx_e = 0;
        float nx_w = 0.f;
        if (item < a.n_items) fetch(item / a.H / a.nP, nx_e0, nx_ne, 0, nx_e, nx_w);
        int nitem = a.n_items;
        for (; item < a.n_items; ++n_item, item = nitem) {
            const int h = item % a.H, bk = item / a.H, kap = bk % a.nP, b = bk / a.nP;
            const int e0 = nx_e0, ne = nx_ne;
            int bat_e = nx_e;
            float bat_w = nx_w;
            {
                const int nn = n_item + 1;
                if ((nn & 31) == 0) load_offsets(nn);
                nitem = __shfl_sync(kAll, my_item, nn & 31);
                nx_e0 = __shfl_sync(kAll, my_e0, nn & 31);
                nx_ne = __shfl_sync(kAll, my_ne, nn & 31);
                if (nitem < a.n_items) fetch(nitem / a.H / a.nP, nx_e0, nx_ne, 0, nx_e, nx_w);
            }
            if (!lane0_wait(&sb.info_empty[inf.i], inf.ph ^ 1u)) break;
            if (lane == 0) {
                ItemInfoB& I = sb.info[inf.i];
                I.b = b; I.kap = kap; I.h = h; I.ne = ne;
                mbar_arrive(&sb.info_full[inf.i]);
            }
            inf.next(kInfo);
            if (ne <= 0) continue;
            if (!lane0_wait(&sb.it_empty[it.i], it.ph ^ 1u)) break;
            if (lane == 0) {
                uint8_t* ib = sm + C::OFF_IT + it.i * C::ITEM_BYTES;
                mbar_arrive_expect_tx(&sb.it_full[it.i], C::ITEM_BYTES);
                for (int sub = 0; sub < HG::SUB; ++sub) {
                    const int off = sub * S * HG::ROW_BYTES;
                    tma_load_2d(ib + off, &tk, &sb.it_full[it.i], h * DH + sub * 64, (b * a.nP + kap) * S);
                    tma_load_2d(ib + C::TILE + off, &tv, &sb.it_full[it.i], h * DH + sub * 64,
                                (b * a.nP + kap) * S);
                }
            }
            it_out[it.i] = true;
            it_ph[it.i] = it.ph;
            it.next(C::IBUF);
            bool ok = true;
            for (int base = 0; base < ne && ok; base += 32) {
                if (base > 0) fetch(b, e0, ne, base, bat_e, bat_w);
                const int my_c = bat_e / a.topk, my_j = bat_e % a.topk;
                const float my_w = bat_w;
                const int cnt = min(32, ne - base);
                for (int u = 0; u < cnt; u += 2) {
                    const int n2 = (u + 1 < cnt) ? 2 : 1;
                    int cc[2], jj[2];
                    float ww[2];
                    for (int x = 0; x < 2; ++x) {
                        const int src = (x < n2) ? u + x : u;
                        cc[x] = __shfl_sync(kAll, my_c, src);
                        jj[x] = __shfl_sync(kAll, my_j, src);
                        ww[x] = __shfl_sync(kAll, my_w, src);
                    }
                    if (!lane0_wait(&sb.st_empty[st.i], st.ph ^ 1u)) { ok = false; break; }
                    if (lane == 0) {
                        uint8_t* stg = sm + C::OFF_ST + st.i * C::STAGE_BYTES;
                        EntryInfo* ei = reinterpret_cast<EntryInfo*>(stg + C::ENT_OFF);
                        mbar_arrive_expect_tx(&sb.st_full[st.i], n2 * C::ENTRY_TX);
                        for (int x = 0; x < n2; ++x) {
                            ei[x].c = cc[x]; ei[x].j = jj[x]; ei[x].w = ww[x];
                            for (int sub = 0; sub < HG::SUB; ++sub) {
                                const int off = (sub * 128 + x * 64) * HG::ROW_BYTES;
                                tma_load_2d(stg + C::Q_OFF + off, &tq, &sb.st_full[st.i], h * DH + sub * 64,
                                            b * a.Lq + cc[x] * S);
                                tma_load_2d(stg + C::DO_OFF + off, &tdo, &sb.st_full[st.i], h * DH + sub * 64,
                                            b * a.Lq + cc[x] * S);
                            }
                            const size_t rb = ((((size_t)b * a.nQ + cc[x]) * a.topk + jj[x]) * a.H + h) * S;
                            tcx::bulk_load(stg + C::VEC_OFF + x * 256, a.lse2_rows + rb, S * 4, &sb.st_full[st.i]);
                            tcx::bulk_load(stg + C::VEC_OFF + 512 + x * 256, a.delta_rows + rb, S * 4,
                                           &sb.st_full[st.i]);
                        }
                    }
                    st_out[st.i] = true;
                    st_ph[st.i] = st.ph;
                    st.next(C::STAGES);
                }
            }
            if (!ok) break;
        }
        if (lane == 0) {
            for (int i = 0; i < C::STAGES; ++i)
                if (st_out[i]) mbar_wait(&sb.st_full[i], st_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < C::IBUF; ++i)
                if (it_out[i]) mbar_wait(&sb.it_full[i], it_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // S = [Q_1; Q_2] K^T and G = [dO_1; dO_2] V^T of each pair (M = 128, N = 64)
        if (lane == 0) {
            Ring st{0, 0}, it{0, 0}, inf{0, 0};
            int q = 0;
            bool issued = false;
            const uint32_t id_s = idesc_bf16(128, S, false, false);
            for (int r = 0; pair_pos(a, r) < a.n_items; ++r) {
                if (!wait(&sb.info_full[inf.i], inf.ph)) break;
                const int ne = sb.info[inf.i].ne;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (ne <= 0) continue;
                const int ng = (ne + 1) >> 1;
                if (!wait(&sb.it_full[it.i], it.ph)) break;
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sm + C::OFF_IT + it.i * C::ITEM_BYTES);
                const uint32_t vaddr = kaddr + C::TILE;
                bool ok = true;
                for (int g = 0; g < ng; ++g) {
                    const int qq = q + g, sbuf = qq & 1;
                    if (!wait(&sb.st_full[st.i], st.ph) || !wait(&sb.s_empty[sbuf], empty_par(qq >> 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t stg = smem_u32(sm + C::OFF_ST + st.i * C::STAGE_BYTES);
                    tcx::mma_kmajor_dh<DH>(tmem + sbuf * C::SGW, stg + C::Q_OFF, 128, kaddr, S, id_s, 0);
                    tcx::mma_kmajor_dh<DH>(tmem + sbuf * C::SGW + 64, stg + C::DO_OFF, 128, vaddr, S, id_s, 0);
                    mma_commit(&sb.s_full[sbuf]);
                    issued = true;
                    st.next(C::STAGES);
                }
                if (!ok) break;
                mma_commit(&sb.it_empty[it.i]);     // K and V are read only by these products
                it.next(C::IBUF);
                q += ng;
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2 || warp == 11) {
        // warp 2: dK += dA^T [Q_1; Q_2], warp 11: dV += (w P)^T [dO_1; dO_2] (M = 64 keys,
        // K = the pair's queries): M = 64 products issue faster from two threads than one
        const bool dvi = warp == 11;
        if (lane == 0) {
            Ring st{0, 0}, inf{0, 0};
            int q = 0, e = 0;
            bool issued = false;
            const uint32_t id_acc = idesc_bf16(64, HG::SUB_COLS, true, true);
            for (int r = 0; pair_pos(a, r) < a.n_items; ++r) {
                if (!wait(&sb.info_full[inf.i], inf.ph)) break;
                const int ne = sb.info[inf.i].ne;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (ne <= 0) continue;
                const int ng = (ne + 1) >> 1;
                const int ob = e % C::NACC;
                if (!wait(&sb.o_empty[ob], empty_par(e / C::NACC))) break;
                tc_fence_after();
                const uint32_t d_dk = tmem + C::COL_ACC + ob * 2 * DH;
                const uint32_t d_dv = d_dk + DH;
                bool ok = true;
                for (int g = 0; g < ng; ++g) {
                    const int qq = q + g, pbuf = qq & 1;
                    const int ksteps = (2 * g + 1 < ne) ? 8 : 4;
                    if (!wait(&sb.p_full[pbuf], full_par(qq >> 1))) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t paddr = smem_u32(sm + C::OFF_P + (C::SHARED_P ? 0 : pbuf * 2 * C::P_BYTES));
                    const uint32_t stg = smem_u32(sm + C::OFF_ST + st.i * C::STAGE_BYTES);
                    if (dvi)
                        tcx::mma_mn_mn_dh<DH>(d_dv, paddr + C::P_BYTES, stg + C::DO_OFF, 128, id_acc, ksteps,
                                              g > 0 ? 1u : 0u);
                    else
                        tcx::mma_mn_mn_dh<DH>(d_dk, paddr, stg + C::Q_OFF, 128, id_acc, ksteps, g > 0 ? 1u : 0u);
                    mma_commit(&sb.st_empty[st.i]);
                    mma_commit(&sb.p_empty[pbuf]);
                    issued = true;
                    st.next(C::STAGES);
                }
                if (!ok) break;
                // the full barrier belongs to the warpgroup that stores this item (item
                // parity), whatever the TMEM buffer: with one accumulator, a barrier
                // shared by both warpgroups could be awaited two phases behind
                mma_commit(&sb.o_full[e & 1]);
                q += ng;
                ++e;
            }
            if (issued) {
                uint64_t* dn = dvi ? &sb.done3 : &sb.done2;
                mma_commit(dn);
                mbar_wait(dn, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp < 11) {
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const int prow = 32 * qd + lane;            // query row of the pair (M = 128 layout)
        const int pe = prow >> 6, ptr = prow & 63;  // its entry and token row
        const int erow = 16 * qd + (lane & 15);     // key row of the dK/dV accumulators (M = 64)
        const int eu = lane >> 4;
        Ring inf{0, 0}, st{0, 0};
        int q = 0, e = 0, n_all = 0, kg = 0;
        const uint64_t nsl2 = tcx::f2_pack(-a.scale_log2, -a.scale_log2);
        for (int r = 0; pair_pos(a, r) < a.n_items; ++r, ++n_all) {
            if (!wait(&sb.info_full[inf.i], inf.ph)) break;
            const ItemInfoB I = sb.info[inf.i];
            mbar_arrive(&sb.info_empty[inf.i]);
            inf.next(kInfo);
            const size_t krow = (size_t)(I.b * a.nP + I.kap) * S + erow;
            __nv_bfloat16* dkrow = a.dk + (krow * a.H + I.h) * DH;
            __nv_bfloat16* dvrow = a.dv + (krow * a.H + I.h) * DH;
            if (I.ne <= 0) {
                if ((n_all & 1) == wg) {
                    tcx::zero_acc_row<64, DH>(dkrow, eu);
                    tcx::zero_acc_row<64, DH>(dvrow, eu);
                }
                continue;
            }
            const int ng = (I.ne + 1) >> 1;
            bool ok = true;
            for (int g = 0; g < ng; ++g) {
                const int qq = q + g;
                const int stage = st.i;
                const uint32_t stph = st.ph;
                st.next(C::STAGES);
                if ((qq & 1) != wg) continue;
                const int sbuf = qq & 1;
                // our own s_full first: its completion implies this pair's stage copy
                // has landed, so the stage barrier's phase below is unambiguous
                if (!wait(&sb.s_full[sbuf], full_par(kg)) || !wait(&sb.st_full[stage], stph)) { ok = false; break; }
                tc_fence_after();
                const uint8_t* stg = sm + C::OFF_ST + stage * C::STAGE_BYTES;
                // a single-entry pair leaves rows 64-127 unused (the products read K = 64)
                const EntryInfo ei = reinterpret_cast<const EntryInfo*>(stg + C::ENT_OFF)[pe];
                const float* vec = reinterpret_cast<const float*>(stg + C::VEC_OFF);
                const float lse2 = vec[pe * 64 + ptr], dlt = vec[128 + pe * 64 + ptr];
                const float wv = ei.w, wsc = wv * a.attn_scale;
                const uint64_t l2 = tcx::f2_pack(lse2, lse2), dl2 = tcx::f2_pack(dlt, dlt);
                const uint64_t wv2 = tcx::f2_pack(wv, wv), wsc2 = tcx::f2_pack(wsc, wsc);
                uint8_t* pa_buf = sm + C::OFF_P + (C::SHARED_P ? 0 : wg * 2 * C::P_BYTES);
                uint8_t* pp_buf = pa_buf + C::P_BYTES;
                const uint32_t ts0 = tmem + lane_base + sbuf * C::SGW;
                const uint32_t tg0 = ts0 + 64;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    // keys 32 hf .. 32 hf + 31 of this query row: S and G columns, one load each
                    uint32_t rx[32], ry[32];
                    tmem_ld_32x32b_x32(ts0 + 32 * hf, rx);
                    tmem_ld_32x32b_x32(tg0 + 32 * hf, ry);
                    tmem_wait_ld();
                    const uint32_t* r0 = rx;
                    const uint32_t* r1 = rx + 16;
                    const uint32_t* r2 = ry;
                    const uint32_t* r3 = ry + 16;
                    if (hf == 1) {
                        tc_fence_before();
                        mbar_arrive(&sb.s_empty[sbuf]);
                    }
                    // key pairs in packed f32x2 arithmetic: p = exp2(-(lse2 - s sl)),
                    // w P and dA = w scale p (g - delta)
                    uint32_t pa[16], pp[16];
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        const uint32_t* rs = p < 8 ? r0 : r1;
                        const uint32_t* rg = p < 8 ? r2 : r3;
                        const int t = 2 * (p & 7);
                        float y0, y1;
                        tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(__uint_as_float(rs[t]), __uint_as_float(rs[t + 1])),
                                                  nsl2, l2), y0, y1);
                        const uint64_t pr2 = tcx::f2_pack(fast_exp2(-y0), fast_exp2(-y1));
                        const uint64_t g2 = tcx::f2_pack(__uint_as_float(rg[t]), __uint_as_float(rg[t + 1]));
                        pp[p] = tcx::pack_bf16x2(tcx::fmul2(pr2, wv2));
                        pa[p] = tcx::pack_bf16x2(tcx::fmul2(tcx::fmul2(pr2, wsc2), tcx::fsub2(g2, dl2)));
                    }
                    if (hf == 0) {
                        // own operand pair: free once this warpgroup's previous pair was read.
                        // Shared pair: pair qq overwrites it once the products of pair qq - 1
                        // (the other warpgroup's) have read it; that barrier completes only for
                        // the other warpgroup's pairs, and its next phase needs this pair's
                        // products, so it is at most one phase from the one awaited.
                        const bool pw = C::SHARED_P
                            ? (qq == 0 || wait(&sb.p_empty[wg ^ 1], full_par((qq - 1) >> 1)))
                            : wait(&sb.p_empty[wg], empty_par(kg));
                        if (!pw) { ok = false; break; }
                    }
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint32_t off = sw128_off(prow, 4 * hf + c4);
                        *reinterpret_cast<uint4*>(pa_buf + off) =
                            make_uint4(pa[4 * c4], pa[4 * c4 + 1], pa[4 * c4 + 2], pa[4 * c4 + 3]);
                        *reinterpret_cast<uint4*>(pp_buf + off) =
                            make_uint4(pp[4 * c4], pp[4 * c4 + 1], pp[4 * c4 + 2], pp[4 * c4 + 3]);
                    }
                }
                if (!ok) break;
                fence_proxy_async_smem();
                mbar_arrive(&sb.p_full[wg]);
                ++kg;
            }
            if (!ok) break;
            q += ng;
            const bool mine = (e & 1) == wg;
            const int ob = e % C::NACC, ko = e >> 1;     // TMEM buffer; this warpgroup's epilogue count
            ++e;
            if (!mine) continue;
            if (!wait(&sb.o_full[wg], full_par(ko))) break;
            tc_fence_after();
            const uint32_t acc = tmem + lane_base + C::COL_ACC + ob * 2 * DH;
            tcx::store_acc_row<64, DH>(acc, dkrow, eu);
            tcx::store_acc_row<64, DH>(acc + DH, dvrow, eu);
            tc_fence_before();
            mbar_arrive(&sb.o_empty[ob]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, CfgP<DH, SHARE>::TMEM_COLS);
    }
}

// ============================================================================ launch
// Dynamic plus static shared memory of each kernel within the 227 KB a CTA may use.
constexpr int kSmemMax = 232448;
template <int S, int DH>
cudaError_t launch_bwd_s(const Shape& sp, const void* q, const void* k, const void* v,
                         const int32_t* idx, const float* w, const float* lse, const void* dout,
                         void* dq, void* dk, void* dv, void* ws, int* status, cudaStream_t st, int* launches) {
    static_assert(CfgA<S, DH>::SMEM + sizeof(BarsA) <= kSmemMax, "shared memory (query-major pass)");
    if constexpr (S == 64) {
        static_assert(CfgP<DH, false>::SMEM + sizeof(BarsB) <= kSmemMax, "shared memory (pair pass)");
        if constexpr (DH == 64)
            static_assert(CfgP<DH, true>::SMEM + sizeof(BarsB) <= kSmemMax, "shared memory (pair pass)");
    }
    else static_assert(CfgK<DH>::SMEM + sizeof(BarsK) <= kSmemMax, "shared memory (key-major pass)");
    CUtensorMap tq, tdo, tk, tv;
    const uint64_t cols = (uint64_t)sp.H * DH;
    constexpr uint32_t bc = tcx::HeadGeom<DH>::SUB_COLS;
    if (!encode_bf16_rows_box(&tq, q, (uint64_t)sp.B * sp.Lq, cols, bc, S) ||
        !encode_bf16_rows_box(&tdo, dout, (uint64_t)sp.B * sp.Lq, cols, bc, S) ||
        !encode_bf16_rows_box(&tk, k, (uint64_t)sp.B * sp.nP * S, cols, bc, S) ||
        !encode_bf16_rows_box(&tv, v, (uint64_t)sp.B * sp.nP * S, cols, bc, S))
        return cudaErrorInvalidValue;
    const BwdWorkspace L = bwd_workspace_layout(sp);
    char* base = static_cast<char*>(ws);
    BwdArgs a;
    a.idx = idx; a.w = w; a.lse = lse;
    a.lse2_rows = reinterpret_cast<float*>(base + L.lse2_off);
    a.delta_rows = reinterpret_cast<float*>(base + L.delta_off);
    a.dwpart = reinterpret_cast<float*>(base + L.dwpart_off);
    a.offset = reinterpret_cast<const int*>(base + L.offset_off);
    a.entry = reinterpret_cast<const int*>(base + L.entry_off);
    a.entry_w = reinterpret_cast<const float*>(base + L.entry_w_off);
    a.order = reinterpret_cast<const int*>(base + L.order_off);
    a.ordered = 0;
    a.dq = static_cast<__nv_bfloat16*>(dq);
    a.dk = static_cast<__nv_bfloat16*>(dk);
    a.dv = static_cast<__nv_bfloat16*>(dv);
    a.status = status;
    a.B = sp.B; a.nQ = sp.nQ; a.nP = sp.nP; a.H = sp.H; a.topk = sp.topk; a.Lq = sp.Lq;
    a.scale_log2 = sp.attn_scale * kLog2e;
    a.attn_scale = sp.attn_scale;
    // pass A stages each item's lse block [S x topk] by TMA when its rows are
    // 16-byte granular and the block fits the per-item staging area
    CUtensorMap tl;
    a.lse_smem = (sp.topk % 4 == 0 && sp.topk <= CfgA<S, DH>::LSE_TOPK_MAX &&
                  (reinterpret_cast<uintptr_t>(lse) & 15) == 0 &&
                  encode_f32_box(&tl, lse, (uint64_t)sp.B * sp.Lq, (uint64_t)sp.H * sp.topk,
                                 (uint32_t)sp.topk, S)) ? 1 : 0;
    if (!a.lse_smem) tl = tq;     // unused placeholder
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

    a.n_items = sp.B * sp.nQ * sp.H;
    auto ka = gca_bwd_q_tc_kernel<S, DH>;
    cudaError_t e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgA<S, DH>::SMEM);
    if (e != cudaSuccess) return e;
    int grid = a.n_items < sms ? a.n_items : sms;
    GCA_LAUNCH("bwd_q_tc", st, ka<<<grid, kThreadsA, CfgA<S, DH>::SMEM, st>>>(tq, tdo, tk, tv, tl, a));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    a.n_items = sp.B * sp.nP * sp.H;
    grid = a.n_items < sms ? a.n_items : sms;
    if constexpr (S == 64) {
        // d = 64: the shared operand pair with two K/V item buffers while an item
        // holds on average at most 12 entries (boundaries frequent), else private pairs
        auto kb = gca_bwd_kv_pair_kernel<DH, false>;
        int smem = CfgP<DH, false>::SMEM;
        if constexpr (DH == 64) {
            if ((long long)sp.nQ * sp.topk <= 12LL * sp.nP) {
                kb = gca_bwd_kv_pair_kernel<DH, true>;
                smem = CfgP<DH, true>::SMEM;
            }
        }
        e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (sp.nP <= 1024) {
            const int* count = reinterpret_cast<const int*>(base + L.count_off);
            GCA_LAUNCH("pair_order", st, pair_order_kernel<<<sp.B, 1024, 0, st>>>(count, sp.nP,
                                                                                    const_cast<int*>(a.order)));
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            *launches += 1;
            a.ordered = 1;
        }
        GCA_LAUNCH("bwd_kv_tc", st, kb<<<grid, kThreadsA, smem, st>>>(tq, tdo, tk, tv, a));
    } else {
        auto kb = gca_bwd_kv128_kernel<DH>;
        e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgK<DH>::SMEM);
        if (e != cudaSuccess) return e;
        GCA_LAUNCH("bwd_kv_tc", st, kb<<<grid, kThreadsA, CfgK<DH>::SMEM, st>>>(tq, tdo, tk, tv, a));
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const Shape& sp, const void* q, const void* k, const void* v,
                          const int32_t* idx, const float* w, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, float* dscore, void* ws, int* status,
                          cudaStream_t st, int* launches) {
    cudaError_t e = launch_inverse_index(sp, idx, w, ws, st, launches);
    if (e != cudaSuccess) return e;
#define GCA_BWD_S(S_, DH_) launch_bwd_s<S_, DH_>(sp, q, k, v, idx, w, lse, dout, dq, dk, dv, ws, status, st, launches)
    if (sp.S == 64) e = sp.d == 32 ? GCA_BWD_S(64, 32) : (sp.d == 128 ? GCA_BWD_S(64, 128) : GCA_BWD_S(64, 64));
    else e = sp.d == 32 ? GCA_BWD_S(128, 32) : (sp.d == 128 ? GCA_BWD_S(128, 128) : GCA_BWD_S(128, 64));
#undef GCA_BWD_S
    if (e != cudaSuccess) return e;
    *launches += 2;
    return launch_dscore(sp, idx, w, ws, dscore, st, launches);
}

}  // namespace gca
