// attn_fwd_tc.cu -- GCA forward on the Blackwell tensor cores (bf16, head
// dimension d = 32, 64 or 128).
//
// GCA (README "Model Architecture"; Figure 1/2; Eq. 2 as the batch form of
// Figure 2): every token t of query chunk c attends separately to each
// retrieved chunk kappa_j (stage 1), O_t^j = softmax(s q_t K_j^T) V_j, and the
// outputs are fused as O_t = sum_j w_j O_t^j (stage 2).  App. B: the forward
// also returns the log-sum-exp of every (token, slot).
//
// Design (one persistent CTA per SM, 11 warps, warp-specialised):
//   warp 0     producer: decodes each work item's retrieval row (valid slots,
//              their weights, codes of empty / out-of-range slots) into a
//              shared-memory info ring, then TMA-loads the Q tile and, for each
//              group of retrieved chunks, their K and V tiles (box 64 x S,
//              128-byte swizzle) straight from the [tokens, H*d] tensors into
//              a ring of stages.
//   warp 1     S issuer (one thread) and TMEM owner: S_g = Q K_g^T for a
//              group of retrieved chunks (N = 128 keys) into one of three
//              TMEM buffers.
//   warp 2     P V issuer (one thread): O += P_g V_g in a TMEM accumulator,
//              A = P_g read from tensor memory.  Two issuers keep either kind
//              of product from waiting behind the other's issue (a
//              tcgen05.mma blocks while the queue drains).
//   warps 3-10 two softmax warpgroups taking alternate groups: read S_g from
//              TMEM, per-slot max / sum / exp2, write P_g = exp(S - m) *
//              (w_j / l_j) as bf16 over the S columns already read (the A
//              operand of the PV MMA), write the lse; each warpgroup also
//              stores O (read from TMEM) for alternate items.
// Because each slot's softmax is normalised before PV and carries its fusion
// weight, the per-slot outputs O_t^j are summed by the tensor core in TMEM
// and never exist in memory.  A work item is (batch row, query chunk, head).
//
// S = 64 : M = 64 MMAs (TMEM rows r at lanes r%16 + 32*(r/16)); a group is two
//          slots; each softmax thread owns one (token, slot) row of 64 keys.
// S = 128: M = 128 MMAs (row r at lane r); a group is one slot; each softmax
//          thread owns one token row of 128 keys.
// Head tiles: d = 64 and 128 as 64-column sub-tiles with the 128-byte swizzle
// (a TMA box each), d = 32 as one 32-column tile with the 64-byte swizzle; the
// score product contracts over every sub-tile, P V issues one N = 64 (or 32)
// product per sub-tile into adjacent TMEM columns.
// Every mbarrier wait is bounded (status GCA_ERR_TIMEOUT, then the CTA winds
// down); indices outside [0, n_pool_chunks) are skipped and reported.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace gca {
namespace {

using namespace tc;

constexpr int kThreads = 352;         // producer, 2 MMA issuers, 2 softmax warpgroups
constexpr int kInfo = 4;                 // item-info ring depth
using tcx::Ring;
using tcx::fast_exp2;
using tcx::pack_bf16;
using tcx::kLog2e;
using tcx::kLn2;

template <int S, int DH>
struct Cfg {
    using G = tcx::HeadGeom<DH>;
    static constexpr int M = S;                         // tokens per item = MMA M
    static constexpr int GS = 128 / S;                  // slots per group
    static constexpr int NG = 128;                      // keys per full group
    // P stays in tensor memory over its own S row (the softmax thread owns the
    // TMEM lane of its row, which is the A operand layout of P V for M = 128 and,
    // row r at lane r % 16 + 32 (r / 16), for M = 64 too), so there are no
    // shared-memory P buffers; an S buffer is then held until its P V products
    // complete.  Three S buffers rotate (two at d = 128, where the O buffers
    // take 256 columns).
    static constexpr bool TP = true;
    static constexpr int NSB = DH == 128 ? 2 : 3;
    // K/V ring depth: what fits beside Q (at S = 64, d = 64 four stages are 1% faster on
    // 16K-token rows with k = 8 and 6% slower on 64K-token rows with k = 16)
    static constexpr int STAGES = TP ? (DH == 32 ? 6 : (DH == 64 ? 5 : 2)) : (DH == 128 ? 2 : 4);
    static constexpr int QBUF = 2;
    static constexpr int TILE = G::tile_bytes(S);       // one slot's K (or V) tile, bytes
    static constexpr int Q_BYTES = G::tile_bytes(S);
    // K half then V half; in each, sub-tile s holds the NG key rows of the
    // group's slots (slot u at rows u*S ..), so a group's K is one B operand
    static constexpr int HALF_BYTES = G::tile_bytes(NG);
    static constexpr int STAGE_BYTES = 2 * HALF_BYTES;
    static constexpr int P_BLOCK = M * 128;             // 64 keys of P for all M rows
    static constexpr int P_BYTES = M * NG * 2;
    static constexpr int VALS = (S == 64) ? 64 : 128;   // S values per softmax thread
    // shared-memory carve-up (all 1024-byte aligned)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + QBUF * Q_BYTES;
    static constexpr int OFF_P = OFF_KV + STAGES * STAGE_BYTES;
    static constexpr int SMEM = OFF_P + (TP ? 0 : 2 * P_BYTES) + 1024;   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;                // NSB S buffers of 128 columns
    static constexpr uint32_t COL_O = NSB * 128;        // two O buffers of DH columns
    static_assert(STAGES <= 6 && NSB <= 3, "barrier arrays");
    static_assert(COL_O + 2 * DH <= TMEM_COLS, "tensor memory");
};

struct FwdArgs {
    const int32_t* idx;
    const float* w;
    __nv_bfloat16* o;
    float* lse;
    int* status;
    int B, nQ, nP, H, topk, Lq;
    float scale_log2;       // attn_scale * log2(e)
    int n_items;
};

struct ItemInfo {
    int b, c, h, n;          // n = valid slots
    int js[kMaxTopk];        // slot number of each valid slot, in slot order
    int kaps[kMaxTopk];      // its retrieved chunk
    float w[kMaxTopk];       // its fusion weight
    int8_t code[kMaxTopk];   // per slot j: 0 valid, 1 empty (-1), 2 outside the pool
};

struct __align__(8) Bars {
    uint64_t info_full[kInfo], info_empty[kInfo];
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[6], kv_empty[6];
    uint64_t s_full[3], s_empty[3];
    uint64_t p_full[4], p_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t done, done2;
    uint32_t tmem;
    int abort;
    ItemInfo info[kInfo];
};

__device__ __forceinline__ bool wait_bar(Bars& sb, uint64_t* bar, uint32_t parity, int* status) {
    return tcx::wait_bar(&sb.abort, bar, parity, status);
}

// Parity to wait for on the k-th use (k = 0, 1, ...) of a buffer: "full"
// barriers complete once per use, "empty" ones start out released.
__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

// P-full barrier of group qq and the phase it completes.  With P in shared
// memory a warpgroup's next P waits for the previous one's products, so one
// barrier per warpgroup suffices.  With P in TMEM nothing holds a fast warp
// back from its warpgroup's next group: its arrival for group qq + 2 could
// then count toward group qq's phase, so each warpgroup alternates two
// barriers (a warp reaches group qq + 4 only after P V of qq + 1 was issued,
// which needed group qq's phase complete).
template <bool TP>
__device__ __forceinline__ int pfull_index(int qq) { return TP ? (qq & 3) : (qq & 1); }
template <bool TP>
__device__ __forceinline__ uint32_t pfull_par(int qq) { return full_par(TP ? (qq >> 2) : (qq >> 1)); }

template <int S, int DH>
__global__ void __launch_bounds__(kThreads, 1)
gca_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
    using C = Cfg<S, DH>;
    using HG = tcx::HeadGeom<DH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ Bars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kInfo; ++i) {
            mbar_init(&sb.info_full[i], 1);
            mbar_init(&sb.info_empty[i], 2 + 256);     // two MMA issuers + every softmax thread
        }
        for (int i = 0; i < C::NSB; ++i) {
            mbar_init(&sb.s_full[i], 1);
            // released by the softmax threads' reads, or (P in TMEM) by the P V products
            mbar_init(&sb.s_empty[i], C::TP ? 1 : 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.q_full[i], 1);
            mbar_init(&sb.q_empty[i], 1);
            mbar_init(&sb.p_full[i], 128);
            mbar_init(&sb.p_full[2 + i], 128);
            mbar_init(&sb.p_empty[i], 1);
            mbar_init(&sb.o_full[i], 1);
            mbar_init(&sb.o_empty[i], 128);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&sb.kv_full[i], 1);
            mbar_init(&sb.kv_empty[i], 1);
        }
        mbar_init(&sb.done, 1);
        mbar_init(&sb.done2, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
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
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            Ring kv{0, 0}, qr{0, 0}, inf{0, 0};
            bool kv_out[6] = {}, q_out[2] = {false, false};
            uint32_t kv_ph[6] = {}, q_ph[2] = {0, 0};
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                const int h = item % a.H, bc = item / a.H, c = bc % a.nQ, b = bc / a.nQ;
                if (!wait_bar(sb, &sb.info_empty[inf.i], inf.ph ^ 1u, a.status)) break;
                ItemInfo& I = sb.info[inf.i];
                const int32_t* row = a.idx + ((size_t)b * a.nQ + c) * a.topk;
                const float* wrow = a.w + ((size_t)b * a.nQ + c) * a.topk;
                int n = 0;
                for (int j = 0; j < a.topk; ++j) {
                    const int kap = row[j];
                    if (kap >= 0 && kap < a.nP) {
                        I.js[n] = j; I.kaps[n] = kap; I.w[n] = wrow[j]; ++n;
                        I.code[j] = 0;
                    } else {
                        I.code[j] = kap < 0 ? 1 : 2;
                        if (kap >= a.nP) set_status(a.status, GCA_ERR_DEVICE_INDEX);
                    }
                }
                I.b = b; I.c = c; I.h = h; I.n = n;
                mbar_arrive(&sb.info_full[inf.i]);
                inf.next(kInfo);
                if (n == 0) continue;
                if (!wait_bar(sb, &sb.q_empty[qr.i], qr.ph ^ 1u, a.status)) break;
                mbar_arrive_expect_tx(&sb.q_full[qr.i], C::Q_BYTES);
                for (int sub = 0; sub < HG::SUB; ++sub)
                    tma_load_2d(sm + C::OFF_Q + qr.i * C::Q_BYTES + sub * S * HG::ROW_BYTES, &tq,
                                &sb.q_full[qr.i], h * DH + sub * 64, b * a.Lq + c * S);
                q_out[qr.i] = true;
                q_ph[qr.i] = qr.ph;
                qr.next(C::QBUF);
                bool ok = true;
                for (int g = 0; g * C::GS < n; ++g) {
                    const int ns = min(C::GS, n - g * C::GS);
                    if (!wait_bar(sb, &sb.kv_empty[kv.i], kv.ph ^ 1u, a.status)) { ok = false; break; }
                    uint8_t* stg = sm + C::OFF_KV + kv.i * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&sb.kv_full[kv.i], ns * 2 * C::TILE);
                    for (int u = 0; u < ns; ++u) {
                        const int y = (b * a.nP + I.kaps[g * C::GS + u]) * S;
                        for (int sub = 0; sub < HG::SUB; ++sub) {
                            const int off = (sub * C::NG + u * S) * HG::ROW_BYTES;
                            tma_load_2d(stg + off, &tk, &sb.kv_full[kv.i], h * DH + sub * 64, y);
                            tma_load_2d(stg + C::HALF_BYTES + off, &tv, &sb.kv_full[kv.i],
                                        h * DH + sub * 64, y);
                        }
                    }
                    kv_out[kv.i] = true;
                    kv_ph[kv.i] = kv.ph;
                    kv.next(C::STAGES);
                }
                if (!ok) break;
            }
            // no copy may still be writing shared memory when the CTA exits
            for (int i = 0; i < C::STAGES; ++i)
                if (kv_out[i]) mbar_wait(&sb.kv_full[i], kv_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < C::QBUF; ++i)
                if (q_out[i]) mbar_wait(&sb.q_full[i], q_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S issuer
        // S_g = Q K_g^T into the S buffer of group g (two, alternating).
        if (lane == 0) {
            Ring kv{0, 0}, qr{0, 0}, inf{0, 0};
            int q = 0;
            bool issued = false;
            const uint32_t id_s128 = idesc_bf16(C::M, 128, false, false);
            const uint32_t id_s64 = idesc_bf16(C::M, 64, false, false);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                if (!wait_bar(sb, &sb.info_full[inf.i], inf.ph, a.status)) break;
                const int n = sb.info[inf.i].n;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (n == 0) continue;
                const int G = (n + C::GS - 1) / C::GS;
                if (!wait_bar(sb, &sb.q_full[qr.i], qr.ph, a.status)) break;
                tc_fence_after();
                const uint32_t qaddr = smem_u32(sm + C::OFF_Q + qr.i * C::Q_BYTES);
                bool ok = true;
                for (int g = 0; g < G; ++g) {
                    const int ns = min(C::GS, n - g * C::GS);
                    const int qq = q + g, sbuf = qq % C::NSB;
                    if (!wait_bar(sb, &sb.kv_full[kv.i], kv.ph, a.status) ||
                        !wait_bar(sb, &sb.s_empty[sbuf], empty_par(qq / C::NSB), a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(sm + C::OFF_KV + kv.i * C::STAGE_BYTES);
                    tcx::mma_kmajor_dh<DH>(tmem + C::COL_S + sbuf * 128, qaddr, S, kaddr, C::NG,
                                           (ns * S == 128) ? id_s128 : id_s64, 0);
                    mma_commit(&sb.s_full[sbuf]);
                    issued = true;
                    kv.next(C::STAGES);
                }
                if (!ok) break;
                mma_commit(&sb.q_empty[qr.i]);     // Q is read only by these products
                qr.next(C::QBUF);
                q += G;
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ P V issuer
        // O += P_g V_g as each softmax warpgroup delivers P_g.
        if (lane == 0) {
            Ring kv{0, 0}, inf{0, 0};
            int q = 0, e = 0;
            bool issued = false;
            const uint32_t id_o = idesc_bf16(C::M, HG::SUB_COLS, false, true);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                if (!wait_bar(sb, &sb.info_full[inf.i], inf.ph, a.status)) break;
                const int n = sb.info[inf.i].n;
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (n == 0) continue;
                const int G = (n + C::GS - 1) / C::GS;
                const int ob = e & 1;
                if (!wait_bar(sb, &sb.o_empty[ob], empty_par(e >> 1), a.status)) break;
                tc_fence_after();
                const uint32_t d_o = tmem + C::COL_O + ob * DH;
                bool ok = true;
                for (int g = 0; g < G; ++g) {
                    const int ns = min(C::GS, n - g * C::GS);
                    const int qq = q + g, pbuf = qq & 1;
                    if (!wait_bar(sb, &sb.p_full[pfull_index<C::TP>(qq)], pfull_par<C::TP>(qq), a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t vaddr = smem_u32(sm + C::OFF_KV + kv.i * C::STAGE_BYTES + C::HALF_BYTES);
                    if constexpr (C::TP) {
                        // P_g sits in its S buffer's first 64 columns (bf16 pairs); a group of
                        // one 64-key slot contracts over its 64 keys only
                        const int sbuf = qq % C::NSB;
                        if (ns * S == 128)
                            tcx::mma_ts_mn_dh<DH, 8>(d_o, tmem + C::COL_S + sbuf * 128, vaddr, C::NG, id_o, g > 0);
                        else
                            tcx::mma_ts_mn_dh<DH, 4>(d_o, tmem + C::COL_S + sbuf * 128, vaddr, C::NG, id_o, g > 0);
                        mma_commit(&sb.kv_empty[kv.i]);
                        mma_commit(&sb.s_empty[sbuf]);
                    } else {
                        const uint32_t paddr = smem_u32(sm + C::OFF_P + pbuf * C::P_BYTES);
                        if (ns * S == 128)
                            tcx::mma_kmajor_mn_dh<DH, 8>(d_o, paddr, C::P_BLOCK, vaddr, C::NG, id_o, g > 0);
                        else
                            tcx::mma_kmajor_mn_dh<DH, 4>(d_o, paddr, C::P_BLOCK, vaddr, C::NG, id_o, g > 0);
                        // S_g is complete (its P exists), so the whole stage may be reused
                        mma_commit(&sb.kv_empty[kv.i]);
                        mma_commit(&sb.p_empty[pbuf]);
                    }
                    issued = true;
                    kv.next(C::STAGES);
                }
                if (!ok) break;
                mma_commit(&sb.o_full[ob]);
                q += G;
                ++e;
            }
            if (issued) {
                mma_commit(&sb.done2);
                mbar_wait(&sb.done2, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wg = (warp - 3) >> 2;                 // warpgroup 0 or 1
        const int qd = warp & 3;
        const int row = (S == 64) ? 16 * qd + (lane & 15) : 32 * qd + lane;
        const int u = (S == 64) ? (lane >> 4) : 0;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        Ring inf{0, 0};
        int q = 0, e = 0, n_all = 0;
        int kg = 0, ko = 0;          // groups / epilogues handled by this warpgroup
        for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++n_all) {
            if (!wait_bar(sb, &sb.info_full[inf.i], inf.ph, a.status)) break;
            const ItemInfo& I = sb.info[inf.i];
            const int b = I.b, c = I.c, h = I.h, n = I.n;
            const size_t tok = (size_t)b * a.Lq + (size_t)c * S + row;
            __nv_bfloat16* orow = a.o + (tok * a.H + h) * DH;
            float* lrow = a.lse ? a.lse + (tok * a.H + h) * a.topk : nullptr;
            // the epilogue of an item is done by one warpgroup, alternating
            const bool my_epi = (n == 0) ? ((n_all & 1) == wg) : ((e & 1) == wg);
            if (my_epi && lrow && u == 0)
                for (int j = 0; j < a.topk; ++j) {
                    const int cd = I.code[j];
                    if (cd == 1) lrow[j] = -INFINITY;
                    else if (cd == 2) lrow[j] = NAN;
                }
            if (n == 0) {
                mbar_arrive(&sb.info_empty[inf.i]);
                inf.next(kInfo);
                if (my_epi) tcx::zero_acc_row<S, DH>(orow, u);
                continue;
            }
            const int G = (n + C::GS - 1) / C::GS;
            bool ok = true;
            for (int g = 0; g < G; ++g) {
                const int qq = q + g;
                if ((qq & 1) != wg) continue;
                const int ns = min(C::GS, n - g * C::GS);
                const bool active = u < ns;
                const int j = active ? I.js[g * C::GS + u] : 0;
                const float wj = active ? I.w[g * C::GS + u] : 0.f;
                const int sbuf = qq % C::NSB;
                if (!wait_bar(sb, &sb.s_full[sbuf], full_par(qq / C::NSB), a.status)) { ok = false; break; }
                tc_fence_after();
                float x[C::VALS];
                const uint32_t taddr = tmem + lane_base + C::COL_S + sbuf * 128;
                float mx, l;
                if constexpr (S == 64) {
                    // the loads return each 16-column chunk's max as well
                    float mc[4];
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci) {
                        uint32_t r[16];
                        mc[ci] = tmem_ld_max_16x32bx2_x16<64>(taddr + 16 * ci, r);
#pragma unroll
                        for (int t = 0; t < 16; ++t) x[16 * ci + t] = __uint_as_float(r[t]);
                    }
                    tmem_wait_ld();
                    if constexpr (!C::TP) {
                        tc_fence_before();
                        mbar_arrive(&sb.s_empty[sbuf]);
                    }
                    // exponentials and the row sum on column pairs (packed f32x2 FMA and
                    // add), four sum chains combined in a fixed order
                    mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
                    const float mb = mx * a.scale_log2;
                    const uint64_t sl2 = tcx::f2_pack(a.scale_log2, a.scale_log2), nmb2 = tcx::f2_pack(-mb, -mb);
                    uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        float y0, y1;
                        tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(x[2 * c], x[2 * c + 1]), sl2, nmb2), y0, y1);
                        x[2 * c] = fast_exp2(y0);
                        x[2 * c + 1] = fast_exp2(y1);
                        acc2[c & 3] = tcx::fadd2(acc2[c & 3], tcx::f2_pack(x[2 * c], x[2 * c + 1]));
                    }
                    float l8[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) tcx::f2_unpack(acc2[u], l8[2 * u], l8[2 * u + 1]);
                    l = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
                } else {
#pragma unroll
                    for (int ci = 0; ci < C::VALS / 16; ++ci) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(taddr + 16 * ci, r);
#pragma unroll
                        for (int t = 0; t < 16; ++t) x[16 * ci + t] = __uint_as_float(r[t]);
                    }
                    tmem_wait_ld();
                    // row max and row sum: eight independent chains, combined in a fixed order
                    float m8[8], l8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
                    for (int i = 8; i < C::VALS; ++i) m8[i & 7] = fmaxf(m8[i & 7], x[i]);
                    mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                    const float mb = mx * a.scale_log2;
#pragma unroll
                    for (int i = 0; i < 8; ++i) l8[i] = 0.f;
#pragma unroll
                    for (int i = 0; i < C::VALS; ++i) {
                        x[i] = fast_exp2(fmaf(x[i], a.scale_log2, -mb));
                        l8[i & 7] += x[i];
                    }
                    l = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
                }
                const float mb = mx * a.scale_log2;
                const float coef = active ? wj / l : 0.f;
                const uint64_t coef2 = tcx::f2_pack(coef, coef);
                if (active && lrow) lrow[j] = (mb + log2f(l)) * kLn2;
                if constexpr (C::TP && S == 128) {
                    // P over the first 64 columns of this row's S buffer, two keys per column
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t pk[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            pk[t] = tcx::pack_bf16(x[32 * ch + 2 * t] * coef, x[32 * ch + 2 * t + 1] * coef);
                        tmem_st_32x32b_x16(taddr + 16 * ch, pk);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                } else if constexpr (C::TP) {
                    // S = 64: P of the group's two slots as one M = 64 A operand over the first
                    // 64 columns of the S buffer (row r at lane r % 16 + 32 (r / 16), as the
                    // score rows): slot u's 64 keys at columns 32 u .. 32 u + 31, written by
                    // the thread that read them (the warp's loads have completed, so the
                    // other slot's scores there are already in registers)
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t pk[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            pk[t] = active ? tcx::pack_bf16x2(tcx::fmul2(tcx::f2_pack(x[32 * ch + 2 * t],
                                                                                  x[32 * ch + 2 * t + 1]), coef2))
                                           : 0u;
                        tmem_st_16x32bx2_x16<32>(taddr + 16 * ch, pk);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                } else {
                    if (!wait_bar(sb, &sb.p_empty[wg], empty_par(kg), a.status)) { ok = false; break; }
                    if (active) {
                        uint8_t* pbase = sm + C::OFF_P + wg * C::P_BYTES + row * 128;
#pragma unroll
                        for (int ch = 0; ch < C::VALS / 8; ++ch) {
                            const int blk = (S == 64) ? u : (ch >> 3);
                            const int cc = ch & 7;
                            *reinterpret_cast<uint4*>(pbase + blk * C::P_BLOCK + ((cc ^ (row & 7)) << 4)) =
                                tcx::pack8x2(x + 8 * ch, coef2);
                        }
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(&sb.p_full[pfull_index<C::TP>(qq)]);
                ++kg;
            }
            mbar_arrive(&sb.info_empty[inf.i]);
            inf.next(kInfo);
            if (!ok) break;
            q += G;
            const bool mine = (e & 1) == wg;
            ++e;
            if (!mine) continue;
            if (!wait_bar(sb, &sb.o_full[wg], full_par(ko), a.status)) break;
            ++ko;
            tc_fence_after();
            const uint32_t oaddr = tmem + lane_base + C::COL_O + wg * DH;
            {
                // O rows of this warp's lanes to registers, release the buffer, then store
                constexpr int NR = (S == 64 ? DH / 2 : DH) / 16;
                uint32_t r[NR][16];
#pragma unroll
                for (int ci = 0; ci < NR; ++ci) {
                    if (S == 64) tmem_ld_16x32bx2_x16<DH / 2>(oaddr + 16 * ci, r[ci]);
                    else tmem_ld_32x32b_x16(oaddr + 16 * ci, r[ci]);
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sb.o_empty[wg]);
                uint4* dst = reinterpret_cast<uint4*>(orow + (S == 64 ? u * (DH / 2) : 0));
#pragma unroll
                for (int ci = 0; ci < NR; ++ci) {
                    dst[2 * ci] = tcx::pack8u(r[ci]);
                    dst[2 * ci + 1] = tcx::pack8u(r[ci] + 8);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg<S, DH>::TMEM_COLS);
    }
}

template <int S, int DH>
cudaError_t launch_s(const Shape& sp, const void* q, const void* k, const void* v,
                     const int32_t* idx, const float* w, void* o, float* lse, int* status,
                     cudaStream_t st) {
    static_assert(Cfg<S, DH>::SMEM + sizeof(Bars) <= 232448, "shared memory: dynamic + static");
    CUtensorMap tq, tk, tv;
    const uint64_t cols = (uint64_t)sp.H * DH;
    constexpr uint32_t bc = tcx::HeadGeom<DH>::SUB_COLS;
    if (!encode_bf16_rows_box(&tq, q, (uint64_t)sp.B * sp.Lq, cols, bc, S) ||
        !encode_bf16_rows_box(&tk, k, (uint64_t)sp.B * sp.nP * S, cols, bc, S) ||
        !encode_bf16_rows_box(&tv, v, (uint64_t)sp.B * sp.nP * S, cols, bc, S))
        return cudaErrorInvalidValue;
    FwdArgs a;
    a.idx = idx; a.w = w; a.o = static_cast<__nv_bfloat16*>(o); a.lse = lse; a.status = status;
    a.B = sp.B; a.nQ = sp.nQ; a.nP = sp.nP; a.H = sp.H; a.topk = sp.topk; a.Lq = sp.Lq;
    a.scale_log2 = sp.attn_scale * kLog2e;
    a.n_items = sp.B * sp.nQ * sp.H;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = a.n_items < sms ? a.n_items : sms;
    auto kern = gca_fwd_tc_kernel<S, DH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<S, DH>::SMEM);
    if (e != cudaSuccess) return e;
    GCA_LAUNCH("fwd_tc", st, kern<<<grid, kThreads, Cfg<S, DH>::SMEM, st>>>(tq, tk, tv, a));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const Shape& sp, const void* q, const void* k, const void* v,
                          const int32_t* idx, const float* w, void* o, float* lse, int* status,
                          cudaStream_t st, int* launches) {
    cudaError_t e;
    if (sp.S == 64) {
        e = sp.d == 32 ? launch_s<64, 32>(sp, q, k, v, idx, w, o, lse, status, st)
          : sp.d == 128 ? launch_s<64, 128>(sp, q, k, v, idx, w, o, lse, status, st)
                        : launch_s<64, 64>(sp, q, k, v, idx, w, o, lse, status, st);
    } else {
        e = sp.d == 32 ? launch_s<128, 32>(sp, q, k, v, idx, w, o, lse, status, st)
          : sp.d == 128 ? launch_s<128, 128>(sp, q, k, v, idx, w, o, lse, status, st)
                        : launch_s<128, 64>(sp, q, k, v, idx, w, o, lse, status, st);
    }
    if (e == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace gca
