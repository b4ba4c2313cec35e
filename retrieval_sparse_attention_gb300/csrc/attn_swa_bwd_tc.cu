// attn_swa_bwd_tc.cu -- backward of the sliding-window causal self-attention
// (the 512-token window self-attention a DRT layer runs before its GCA
// module; paper summary sections 1 and 4.1.2) on the Blackwell tensor cores
// (bf16, d = 64).
//
// With p_ts = exp(attn_scale q_t . k_s - lse_t) over the window of t,
// delta_t = dO_t . O_t, dp_ts = dO_t . v_s and ds_ts = attn_scale p_ts (dp_ts - delta_t):
//   dQ_t = sum_s ds_ts k_s,   dK_s = sum_t ds_ts q_t,   dV_s = sum_t p_ts dO_t.
// Two launches, no atomics (every output row is written by one CTA):
//   pass A  query-major, item = (batch row, 128-token query tile, head).  The
//           item's Q, dO and O tiles land once; each math thread forms delta_t
//           of its token row from the dO and O rows in shared memory, and the
//           item's storing warpgroup writes -lse_t log2(e) and -attn_scale
//           delta_t as [B, H, Lp] rows for pass B.  Unit = one 64-key tile:
//           S = Q K^T and dP = dO V^T (M = 128 tokens, N = 64 keys) into a
//           128-column TMEM buffer.  A math thread owns token row t, which is
//           TMEM lane t -- the layout of an A operand -- so it writes ds (bf16
//           pairs) over the S columns it has read and dQ += dS K reads A from
//           tensor memory.
//   pass B  key-major, item = (batch row, 128-key tile, head).  Unit = 64
//           queries, half of a 128-query stage that also carries those queries'
//           two pass-A rows: S^T = K Q^T and dP^T = V dO^T (M = 128 keys); a math
//           thread owns key row s, writes dS^T over S^T and P^T over dP^T, and
//           dK += dS^T Q, dV += P^T dO read A from tensor memory (two issuing
//           threads).
// In both passes the two math warpgroups take alternate units of the same
// item, three TMEM buffers rotate, the accumulation products release a buffer
// when they have read it, and no shared-memory operand buffer exists.
// A CTA walks a contiguous run of items, tile index fastest, so consecutive
// items of a (batch row, head) strip share most of their units' tiles (K/V
// tiles in pass A, Q/dO stages in pass B): a shared tile stays in its ring
// slot and only the new ones are loaded (2 of 10 K/V tiles, 1 of 5 stages at
// W = 512).  Slots are filled and released in load order; the host checks for
// the window at hand that no item waits for a slot a later item still holds,
// and otherwise every item loads all its tiles.  Tensor maps are 3-D over
// [B, L, H*d], so rows past a sequence end read as zeros; output rows past it
// are never written.  Every mbarrier wait is bounded.
#include <math.h>

#include <vector>

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
using tcx::Ring;

constexpr int BM = 128;                  // item rows = MMA M
constexpr int BT = 64;                   // unit width = MMA N of the score products
constexpr int TILE128 = 128 * 128;       // 128 rows x 64 bf16
constexpr int TILE64 = 64 * 128;         // 64 rows x 64 bf16
// Tensor memory: an X ring of 64-column slots holds a unit's S (S^T) and then
// the bf16 operands the math writes over it, until the accumulation products
// have read them; a Y ring holds its dP (dP^T) and is free as soon as the math
// has read it; the accumulators follow.
constexpr int NX = 4;
constexpr int NY = 2;
constexpr uint32_t COL_X = 0;
constexpr uint32_t COL_Y = NX * 64;
constexpr uint32_t COL_ACC = COL_Y + NY * 64;
constexpr uint32_t TMEM_COLS = 512;
static_assert(COL_ACC + 128 <= TMEM_COLS, "tensor memory");
constexpr int kSmemMax = 232448;

struct SwaBwdArgs {
    const float* lse;        // [B, L, H] (forward output)
    float* nlse2T;           // [B, H, Lp]: -lse * log2(e)       (written by pass A)
    float* ndscT;            // [B, H, Lp]: -attn_scale * delta  (written by pass A)
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int* status;
    int B, L, H, W, Lp;
    int nQT, nKT;            // 128-token query tiles, 128-key tiles per row
    float scale_log2;        // attn_scale * log2(e)
    float scale;             // attn_scale
    int n_items;
    int chunk;               // items per CTA (a contiguous run)
    int slide;               // keep shared tiles of consecutive items resident
};

// Ring bookkeeping shared by the producer and the consumers of a ring whose
// entries are the tiles of items (k0 .. k1 per item, increasing within a strip).
// Ring position of a tile = the order in which it was loaded; slot = position
// % NSLOT.  begin() returns the first tile of the item that must be loaded:
// k0, or the one after the last tile of the previous item when that item kept
// its tiles k0 .. for this one.
struct Slide {
    int strip, klast, nload;
    __device__ __forceinline__ int begin(bool kept, int strip_, int k0, int k1) {
        const int from = (kept && strip_ == strip && k0 <= klast + 1) ? klast + 1 : k0;
        nload += k1 - from + 1;
        klast = k1;
        strip = strip_;
        return from;
    }
    __device__ __forceinline__ int pos(int k1, int k) const { return nload - 1 - (k1 - k); }
};

__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

// A global load issued where it stands: the compiler may not sink it to the
// value's first use (an item later), so its latency overlaps a whole item.
__device__ __forceinline__ float ld_early(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// 64 fp32 accumulator columns of this thread's lane -> 32 bf16 pairs (the TMEM
// reads are warp-collective).
__device__ __forceinline__ void load_row64(uint32_t taddr, uint32_t (&pk)[32]) {
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr + 16 * ci, r);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 8; ++u)
            pk[8 * ci + u] = tcx::pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
    }
}
__device__ __forceinline__ void store_row64(__nv_bfloat16* dst, const uint32_t (&pk)[32]) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c) d4[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}

// ============================================================================ pass A (dQ, delta)
namespace pa {
constexpr int kThreads = 384;                    // producer, S, dQ and dP issuers, 8 math warps
constexpr int IBUF = 2;
constexpr int ITEM = 3 * TILE128;                // Q, dO, O
// the producer issues the next item's buffer (and its lse load) an item ahead, so a
// single item buffer would wait on its own item: the protocol needs two
static_assert(IBUF == 2, "pass A needs two item buffers");
constexpr int NSLOT = 8;                         // K/V tile slots
constexpr int SLOT = 2 * TILE64;                 // K, V
constexpr int OFF_IT = 0;
constexpr int OFF_KV = IBUF * ITEM;
constexpr int SMEM = OFF_KV + NSLOT * SLOT + 1024;

struct Item {
    int b, qt, h, strip, k0, k1;     // 64-key tiles k0 .. k1
};
// item = (b * H + h) * nQT + qt
__device__ __forceinline__ Item decode(const SwaBwdArgs& a, int item) {
    Item it;
    it.qt = item % a.nQT;
    it.strip = item / a.nQT;
    it.h = it.strip % a.H;
    it.b = it.strip / a.H;
    int lo = it.qt * BM - a.W + 1;
    if (lo < 0) lo = 0;
    it.k0 = lo / BT;
    it.k1 = (it.qt * BM + BM - 1) / BT;
    return it;
}
// Does this item keep its tiles k >= next.k0 resident for the next item of the run?
__device__ __forceinline__ bool keeps(const SwaBwdArgs& a, const Item& I, int item, int c1, Item& nx) {
    if (!a.slide || item + 1 >= c1) return false;
    nx = decode(a, item + 1);
    return nx.strip == I.strip;
}

struct __align__(8) Bars {
    uint64_t it_full[IBUF], it_empty[IBUF];
    uint64_t kv_full[NSLOT], kv_empty[NSLOT];
    uint64_t x_full[NX], x_empty[NX], y_empty[NY];
    uint64_t p_full[4];                  // per unit, cycling four (two per warpgroup)
    uint64_t o_full[2], o_empty[2];      // per dQ accumulator = per storing warpgroup
    uint64_t done, done2, done3;
    uint32_t tmem;
    int abort;
};
static_assert(SMEM + sizeof(Bars) <= kSmemMax, "shared memory (pass A)");

__global__ void __launch_bounds__(kThreads, 1)
swa_bwd_q_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap to, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const SwaBwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ Bars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };
    const int c0 = static_cast<int>((long long)blockIdx.x * a.n_items / gridDim.x);
    const int c1 = static_cast<int>((long long)(blockIdx.x + 1) * a.n_items / gridDim.x);

    if (threadIdx.x == 0) {
        for (int i = 0; i < IBUF; ++i) {
            mbar_init(&sb.it_full[i], 1);
            mbar_init(&sb.it_empty[i], 2 + 256);      // the S and dP issuers + every math thread
        }
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&sb.kv_full[i], 1);
            mbar_init(&sb.kv_empty[i], 1);
        }
        for (int i = 0; i < NX; ++i) {
            mbar_init(&sb.x_full[i], 2);              // the S and the dP products
            mbar_init(&sb.x_empty[i], 1);
        }
        for (int i = 0; i < NY; ++i) mbar_init(&sb.y_empty[i], 128);
        for (int i = 0; i < 4; ++i) mbar_init(&sb.p_full[i], 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.o_full[i], 1);
            mbar_init(&sb.o_empty[i], 128);
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
        prefetch_tmap(&to);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 1) {
        tmem_alloc(&sb.tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            Ring it{0, 0};
            Slide sl{-1, -1, 0};
            bool kept = false;
            bool kv_out[NSLOT] = {}, it_out[IBUF] = {};
            uint32_t kv_ph[NSLOT] = {}, it_ph[IBUF] = {};
            bool ok = true;
            // Q, dO and O of an item: issued one item ahead, before the item's new K/V
            // tiles (whose slots the item's own first units free)
            auto load_item = [&](int item) {
                const Item J = decode(a, item);
                if (!wait(&sb.it_empty[it.i], it.ph ^ 1u)) return false;
                uint8_t* ib = sm + OFF_IT + it.i * ITEM;
                mbar_arrive_expect_tx(&sb.it_full[it.i], 3 * TILE128);
                tma_load_3d(ib, &tq, &sb.it_full[it.i], J.h * 64, J.qt * BM, J.b);
                tma_load_3d(ib + TILE128, &tdo, &sb.it_full[it.i], J.h * 64, J.qt * BM, J.b);
                tma_load_3d(ib + 2 * TILE128, &to, &sb.it_full[it.i], J.h * 64, J.qt * BM, J.b);
                it_out[it.i] = true;
                it_ph[it.i] = it.ph;
                it.next(IBUF);
                return true;
            };
            if (c0 < c1) ok = load_item(c0);
            for (int item = c0; item < c1 && ok; ++item) {
                const Item I = decode(a, item);
                Item nx;
                const bool keep = keeps(a, I, item, c1, nx);
                if (item + 1 < c1 && !load_item(item + 1)) break;
                const int from = sl.begin(kept, I.strip, I.k0, I.k1);
                for (int k = from; k <= I.k1; ++k) {
                    const int p = sl.pos(I.k1, k), slot = p % NSLOT;
                    const uint32_t ph = static_cast<uint32_t>(p / NSLOT) & 1u;
                    if (!wait(&sb.kv_empty[slot], ph ^ 1u)) { ok = false; break; }
                    uint8_t* kv = sm + OFF_KV + slot * SLOT;
                    mbar_arrive_expect_tx(&sb.kv_full[slot], 2 * TILE64);
                    tma_load_3d(kv, &tk, &sb.kv_full[slot], I.h * 64, k * BT, I.b);
                    tma_load_3d(kv + TILE64, &tv, &sb.kv_full[slot], I.h * 64, k * BT, I.b);
                    kv_out[slot] = true;
                    kv_ph[slot] = ph;
                }
                kept = keep;
            }
            for (int i = 0; i < NSLOT; ++i)
                if (kv_out[i]) mbar_wait(&sb.kv_full[i], kv_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < IBUF; ++i)
                if (it_out[i]) mbar_wait(&sb.it_full[i], it_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1 || warp == 11) {
        // ------------------------------------------------------------ warp 1: S = Q K^T, warp 11: dP = dO V^T
        // (two issuing threads: one thread issues at most one MMA per ~46 cycles)
        const bool dpi = warp == 11;
        if (lane == 0) {
            Ring it{0, 0};
            Slide sl{-1, -1, 0};
            bool kept = false;
            int u = 0;
            bool issued = false, ok = true;
            const uint32_t id_s = idesc_bf16(BM, BT, false, false);
            for (int item = c0; item < c1 && ok; ++item) {
                const Item I = decode(a, item);
                Item nx;
                const bool keep = keeps(a, I, item, c1, nx);
                sl.begin(kept, I.strip, I.k0, I.k1);
                kept = keep;
                if (!wait(&sb.it_full[it.i], it.ph)) break;
                // A = Q (S) or dO (dP); B = the K or V tile
                const uint32_t aaddr = smem_u32(sm + OFF_IT + it.i * ITEM) + (dpi ? TILE128 : 0);
                for (int k = I.k0; k <= I.k1; ++k, ++u) {
                    const int p = sl.pos(I.k1, k), slot = p % NSLOT;
                    const int xs = u % NX, ys = u % NY;
                    if (!wait(&sb.kv_full[slot], static_cast<uint32_t>(p / NSLOT) & 1u) ||
                        !(dpi ? wait(&sb.y_empty[ys], empty_par(u / NY)) : wait(&sb.x_empty[xs], empty_par(u / NX)))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t baddr = smem_u32(sm + OFF_KV + slot * SLOT) + (dpi ? TILE64 : 0);
                    tcx::mma_kmajor_k64(dpi ? tmem + COL_Y + ys * 64 : tmem + COL_X + xs * 64, aaddr, baddr, id_s, 0);
                    mma_commit(&sb.x_full[xs]);
                    issued = true;
                }
                if (!ok) break;
                mma_commit(&sb.it_empty[it.i]);       // Q (dO) is read only by these products
                it.next(IBUF);
            }
            if (issued) {
                uint64_t* dn = dpi ? &sb.done3 : &sb.done;
                mma_commit(dn);
                mbar_wait(dn, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ dQ += dS K (A from TMEM)
        if (lane == 0) {
            Slide sl{-1, -1, 0};
            bool kept = false;
            int u = 0, e = 0;
            bool issued = false, ok = true;
            const uint32_t id_acc = idesc_bf16(BM, 64, false, true);
            for (int item = c0; item < c1 && ok; ++item, ++e) {
                const Item I = decode(a, item);
                Item nx;
                const bool keep = keeps(a, I, item, c1, nx);
                sl.begin(kept, I.strip, I.k0, I.k1);
                kept = keep;
                const int ob = e & 1;
                if (!wait(&sb.o_empty[ob], empty_par(e >> 1))) break;
                tc_fence_after();
                for (int k = I.k0; k <= I.k1; ++k, ++u) {
                    const int slot = sl.pos(I.k1, k) % NSLOT;
                    const int xs = u % NX;
                    if (!wait(&sb.p_full[u & 3], full_par(u >> 2))) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(sm + OFF_KV + slot * SLOT);
                    tcx::mma_ts_mn_dh<64, 4>(tmem + COL_ACC + ob * 64, tmem + COL_X + xs * 64, kaddr, BT, id_acc,
                                             k > I.k0 ? 1u : 0u);
                    mma_commit(&sb.x_empty[xs]);
                    // the tile's last product (S, dP complete before ds exists): release
                    // it unless the next item of the run uses it too
                    if (!keep || k < nx.k0) mma_commit(&sb.kv_empty[slot]);
                    issued = true;
                }
                if (!ok) break;
                mma_commit(&sb.o_full[ob]);
            }
            if (issued) {
                mma_commit(&sb.done2);
                mbar_wait(&sb.done2, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp < 11) {
        // ------------------------------------------------------------ math warpgroups
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const int row = 32 * qd + lane;               // token row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const uint32_t span = static_cast<uint32_t>(a.W - 1);
        const uint64_t sl2 = tcx::f2_pack(a.scale_log2, a.scale_log2);
        const uint64_t sc2 = tcx::f2_pack(a.scale, a.scale);
        // lse of this thread's row of an item (rows past L read row L - 1; unused)
        auto lse_of = [&](int item) {
            const Item J = decode(a, item);
            const int t = min(J.qt * BM + row, a.L - 1);
            return ld_early(a.lse + ((size_t)J.b * a.L + t) * a.H + J.h);
        };
        Ring it{0, 0};
        int u = 0, e = 0;
        bool ok = true;
        float lse_next = c0 < c1 ? lse_of(c0) : 0.f;
        // the dQ epilogue of an item this warpgroup stores runs after its first unit
        // of the next item, so the wait for the item's last product overlaps work
        int pend_e = -1;
        __nv_bfloat16* pend_dst = nullptr;
        bool pend_live = false;
        auto epilogue = [&]() {
            if (!wait(&sb.o_full[wg], full_par(pend_e >> 1))) return false;
            tc_fence_after();
            uint32_t pk[32];
            load_row64(tmem + lane_base + COL_ACC + wg * 64, pk);
            tc_fence_before();
            mbar_arrive(&sb.o_empty[wg]);
            if (pend_live) store_row64(pend_dst, pk);
            pend_e = -1;
            return true;
        };
        for (int item = c0; item < c1 && ok; ++item, ++e) {
            const Item I = decode(a, item);
            const int t0 = I.qt * BM;
            const int t = t0 + row;
            const bool live = t < a.L;
            // this row's lse was loaded one item ahead; start the next one's load
            const float nl2 = live ? -lse_next * kLog2e : 0.f;
            if (item + 1 < c1) lse_next = lse_of(item + 1);
            if (!wait(&sb.it_full[it.i], it.ph)) break;
            // delta_t = dO_t . O_t from this row of the two tiles (128-byte swizzled rows)
            float dlt;
            {
                const uint8_t* ib = sm + OFF_IT + it.i * ITEM;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t off = tcx::sw128_off(row, c);
                    const uint4 g4 = *reinterpret_cast<const uint4*>(ib + TILE128 + off);
                    const uint4 o4 = *reinterpret_cast<const uint4*>(ib + 2 * TILE128 + off);
                    const __nv_bfloat162* hg = reinterpret_cast<const __nv_bfloat162*>(&g4);
                    const __nv_bfloat162* ho = reinterpret_cast<const __nv_bfloat162*>(&o4);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float2 fg = __bfloat1622float2(hg[v]), fo = __bfloat1622float2(ho[v]);
                        acc[2 * v] = fmaf(fg.x, fo.x, acc[2 * v]);
                        acc[2 * v + 1] = fmaf(fg.y, fo.y, acc[2 * v + 1]);
                    }
                }
                dlt = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            }
            mbar_arrive(&sb.it_empty[it.i]);
            it.next(IBUF);
            const float ndsc = -dlt * a.scale;
            const bool mine = (e & 1) == wg;
            if (mine) {
                const size_t vrow = ((size_t)I.b * a.H + I.h) * a.Lp + t;    // t < Lp
                a.nlse2T[vrow] = nl2;
                a.ndscT[vrow] = live ? ndsc : 0.f;
            }
            const uint64_t nl22 = tcx::f2_pack(nl2, nl2), ndsc2 = tcx::f2_pack(ndsc, ndsc);
            const int lo = t - a.W + 1;
            for (int k = I.k0; k <= I.k1; ++k, ++u) {
                if ((u & 1) != wg) continue;
                const int xs = u % NX, ys = u % NY;
                if (!wait(&sb.x_full[xs], full_par(u / NX))) { ok = false; break; }
                tc_fence_after();
                const int kbase = k * BT;
                // warpgroup-uniform: does the window edge or the diagonal cross this tile?
                const bool edge = kbase + BT - 1 > t0 || kbase < t0 + BM - a.W;
                const uint32_t xb = tmem + lane_base + COL_X + xs * 64;
                const uint32_t yb = tmem + lane_base + COL_Y + ys * 64;
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
                    // keys kbase + 32 pc .. + 31: S (X columns 32 pc ..) and dP (Y columns 32 pc ..)
                    uint32_t r0[16], r1[16], r2[16], r3[16];
                    tmem_ld_32x32b_x16(xb + 32 * pc, r0);
                    tmem_ld_32x32b_x16(xb + 32 * pc + 16, r1);
                    tmem_ld_32x32b_x16(yb + 32 * pc, r2);
                    tmem_ld_32x32b_x16(yb + 32 * pc + 16, r3);
                    tmem_wait_ld();
                    if (pc == 1) {                                // dP fully read: free its slot
                        tc_fence_before();
                        mbar_arrive(&sb.y_empty[ys]);
                    }
                    const int cb = kbase + 32 * pc - lo;          // column 0 relative to lo
                    uint32_t pk[16];
                    auto body = [&](bool msk) {
#pragma unroll
                        for (int p2 = 0; p2 < 16; ++p2) {
                            const uint32_t* rs = p2 < 8 ? r0 : r1;
                            const uint32_t* rg = p2 < 8 ? r2 : r3;
                            const int tt = 2 * (p2 & 7);
                            float y0, y1;
                            tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(__uint_as_float(rs[tt]), __uint_as_float(rs[tt + 1])),
                                                      sl2, nl22), y0, y1);
                            float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
                            if (msk) {
                                p0 = static_cast<uint32_t>(cb + 2 * p2) > span ? 0.f : p0;
                                p1 = static_cast<uint32_t>(cb + 2 * p2 + 1) > span ? 0.f : p1;
                            }
                            const uint64_t gd = tcx::ffma2(
                                tcx::f2_pack(__uint_as_float(rg[tt]), __uint_as_float(rg[tt + 1])), sc2, ndsc2);
                            pk[p2] = tcx::pack_bf16x2(tcx::fmul2(tcx::f2_pack(p0, p1), gd));
                        }
                    };
                    if (edge) body(true);
                    else body(false);
                    // dS over S columns 16 pc .. 16 pc + 15 (already read)
                    tmem_st_32x32b_x16(xb + 16 * pc, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sb.p_full[u & 3]);
                if (pend_e >= 0 && !epilogue()) { ok = false; break; }
            }
            if (!ok) break;
            if (mine) {
                pend_e = e;
                pend_dst = a.dq + (((size_t)I.b * a.L + t) * a.H + I.h) * 64;
                pend_live = live;
            }
        }
        if (ok && pend_e >= 0) epilogue();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}
}  // namespace pa

// ============================================================================ pass B (dK, dV)
namespace pb {
constexpr int kThreads = 384;                    // + warp 11: the dV issuer
constexpr int IBUF = 2;
constexpr int ITEM = 2 * TILE128;                // K, V
static_assert(IBUF == 2, "pass B needs two item buffers (one item of lead)");
constexpr int VEC_OFF = 2 * TILE128;             // after the Q and dO tiles: nlse2[128], ndsc[128]
constexpr int SLOT = VEC_OFF + 1024;             // one 128-query stage
constexpr int NSLOT = 4;
constexpr int OFF_IT = 0;
constexpr int OFF_ST = IBUF * ITEM;
constexpr int SMEM = OFF_ST + NSLOT * SLOT + 1024;

struct Item {
    int b, kt, h, strip, g0, g1;     // 128-query stages g0 .. g1
};
// item = (b * H + h) * nKT + kt
__device__ __forceinline__ Item decode(const SwaBwdArgs& a, int item) {
    Item it;
    it.kt = item % a.nKT;
    it.strip = item / a.nKT;
    it.h = it.strip % a.H;
    it.b = it.strip / a.H;
    it.g0 = it.kt;
    int last = it.kt * BM + BM - 1 + a.W - 1;            // last query that sees a key of the tile
    if (last > a.L - 1) last = a.L - 1;
    it.g1 = last / BM;
    return it;
}
__device__ __forceinline__ bool keeps(const SwaBwdArgs& a, const Item& I, int item, int c1, Item& nx) {
    if (!a.slide || item + 1 >= c1) return false;
    nx = decode(a, item + 1);
    return nx.strip == I.strip;
}

struct __align__(8) Bars {
    uint64_t it_full[IBUF], it_empty[IBUF];
    uint64_t st_full[NSLOT], st_empty[NSLOT];
    uint64_t x_full[NX], x_empty[NX], y_empty[NY];
    uint64_t p_full[4];
    uint64_t o_full[2], o_empty;         // o_full per storing warpgroup
    uint64_t done, done2, done3;
    uint32_t tmem;
    int abort;
};
static_assert(SMEM + sizeof(Bars) <= kSmemMax, "shared memory (pass B)");

__global__ void __launch_bounds__(kThreads, 1)
swa_bwd_kv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const SwaBwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ Bars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };
    const int c0 = static_cast<int>((long long)blockIdx.x * a.n_items / gridDim.x);
    const int c1 = static_cast<int>((long long)(blockIdx.x + 1) * a.n_items / gridDim.x);

    if (threadIdx.x == 0) {
        for (int i = 0; i < IBUF; ++i) {
            mbar_init(&sb.it_full[i], 1);
            mbar_init(&sb.it_empty[i], 1);
        }
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&sb.st_full[i], 1);
            mbar_init(&sb.st_empty[i], 2);            // the dK and the dV issuer
        }
        for (int i = 0; i < NX; ++i) {
            mbar_init(&sb.x_full[i], 1);
            mbar_init(&sb.x_empty[i], 2);            // the dK and the dV issuer
        }
        for (int i = 0; i < NY; ++i) mbar_init(&sb.y_empty[i], 128);
        for (int i = 0; i < 4; ++i) mbar_init(&sb.p_full[i], 128);
        mbar_init(&sb.o_full[0], 2);
        mbar_init(&sb.o_full[1], 2);
        mbar_init(&sb.o_empty, 128);
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
        tmem_alloc(&sb.tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            Ring it{0, 0};
            Slide sl{-1, -1, 0};
            bool kept = false;
            bool st_out[NSLOT] = {}, it_out[IBUF] = {};
            uint32_t st_ph[NSLOT] = {}, it_ph[IBUF] = {};
            bool ok = true;
            // K and V of an item: issued one item ahead, before the item's new stages
            // (whose slots the item's own first units free)
            auto load_item = [&](int item) {
                const Item J = decode(a, item);
                if (!wait(&sb.it_empty[it.i], it.ph ^ 1u)) return false;
                uint8_t* ib = sm + OFF_IT + it.i * ITEM;
                mbar_arrive_expect_tx(&sb.it_full[it.i], 2 * TILE128);
                tma_load_3d(ib, &tk, &sb.it_full[it.i], J.h * 64, J.kt * BM, J.b);
                tma_load_3d(ib + TILE128, &tv, &sb.it_full[it.i], J.h * 64, J.kt * BM, J.b);
                it_out[it.i] = true;
                it_ph[it.i] = it.ph;
                it.next(IBUF);
                return true;
            };
            if (c0 < c1) ok = load_item(c0);
            for (int item = c0; item < c1 && ok; ++item) {
                const Item I = decode(a, item);
                Item nx;
                const bool keep = keeps(a, I, item, c1, nx);
                if (item + 1 < c1 && !load_item(item + 1)) break;
                const size_t vbase = ((size_t)I.b * a.H + I.h) * a.Lp;
                const int from = sl.begin(kept, I.strip, I.g0, I.g1);
                for (int g = from; g <= I.g1; ++g) {
                    const int p = sl.pos(I.g1, g), slot = p % NSLOT;
                    const uint32_t ph = static_cast<uint32_t>(p / NSLOT) & 1u;
                    if (!wait(&sb.st_empty[slot], ph ^ 1u)) { ok = false; break; }
                    uint8_t* stg = sm + OFF_ST + slot * SLOT;
                    const int qb = g * BM;
                    mbar_arrive_expect_tx(&sb.st_full[slot], 2 * TILE128 + 2 * BM * 4);
                    tma_load_3d(stg, &tq, &sb.st_full[slot], I.h * 64, qb, I.b);
                    tma_load_3d(stg + TILE128, &tdo, &sb.st_full[slot], I.h * 64, qb, I.b);
                    tcx::bulk_load(stg + VEC_OFF, a.nlse2T + vbase + qb, BM * 4, &sb.st_full[slot]);
                    tcx::bulk_load(stg + VEC_OFF + BM * 4, a.ndscT + vbase + qb, BM * 4, &sb.st_full[slot]);
                    st_out[slot] = true;
                    st_ph[slot] = ph;
                }
                kept = keep;
            }
            for (int i = 0; i < NSLOT; ++i)
                if (st_out[i]) mbar_wait(&sb.st_full[i], st_ph[i], nullptr, 100000000ull);
            for (int i = 0; i < IBUF; ++i)
                if (it_out[i]) mbar_wait(&sb.it_full[i], it_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S^T = K Q^T, dP^T = V dO^T
        if (lane == 0) {
            Ring it{0, 0};
            Slide sl{-1, -1, 0};
            bool kept = false;
            int u = 0;
            bool issued = false, ok = true;
            const uint32_t id_s = idesc_bf16(BM, BT, false, false);
            for (int item = c0; item < c1 && ok; ++item) {
                const Item I = decode(a, item);
                Item nx;
                const bool keep = keeps(a, I, item, c1, nx);
                sl.begin(kept, I.strip, I.g0, I.g1);
                kept = keep;
                if (!wait(&sb.it_full[it.i], it.ph)) break;
                const uint32_t kaddr = smem_u32(sm + OFF_IT + it.i * ITEM);
                const uint32_t vaddr = kaddr + TILE128;
                for (int g = I.g0; g <= I.g1 && ok; ++g) {
                    const int p = sl.pos(I.g1, g), slot = p % NSLOT;
                    if (!wait(&sb.st_full[slot], static_cast<uint32_t>(p / NSLOT) & 1u)) { ok = false; break; }
                    const uint32_t qaddr = smem_u32(sm + OFF_ST + slot * SLOT);
                    for (int hf = 0; hf < 2; ++hf, ++u) {
                        const int xs = u % NX, ys = u % NY;
                        if (!wait(&sb.x_empty[xs], empty_par(u / NX)) || !wait(&sb.y_empty[ys], empty_par(u / NY))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        tcx::mma_kmajor_k64(tmem + COL_X + xs * 64, kaddr, qaddr + hf * TILE64, id_s, 0);
                        tcx::mma_kmajor_k64(tmem + COL_Y + ys * 64, vaddr, qaddr + TILE128 + hf * TILE64, id_s, 0);
                        mma_commit(&sb.x_full[xs]);
                        issued = true;
                    }
                }
                if (!ok) break;
                mma_commit(&sb.it_empty[it.i]);       // K and V are read only by these products
                it.next(IBUF);
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2 || warp == 11) {
        // warp 2: dK += dS^T Q, warp 11: dV += P^T dO (A from TMEM, K = 64 queries)
        const bool dvi = warp == 11;
        if (lane == 0) {
            Slide sl{-1, -1, 0};
            bool kept = false;
            int u = 0, e = 0;
            bool issued = false, ok = true;
            const uint32_t id_acc = idesc_bf16(BM, 64, false, true);
            const uint32_t d_acc = tmem + COL_ACC + (dvi ? 64 : 0);
            for (int item = c0; item < c1 && ok; ++item, ++e) {
                const Item I = decode(a, item);
                Item nx;
                const bool keep = keeps(a, I, item, c1, nx);
                sl.begin(kept, I.strip, I.g0, I.g1);
                kept = keep;
                if (!wait(&sb.o_empty, empty_par(e))) break;
                tc_fence_after();
                for (int g = I.g0; g <= I.g1 && ok; ++g) {
                    const int slot = sl.pos(I.g1, g) % NSLOT;
                    const uint32_t xaddr = smem_u32(sm + OFF_ST + slot * SLOT) + (dvi ? TILE128 : 0);
                    for (int hf = 0; hf < 2; ++hf, ++u) {
                        const int xs = u % NX;
                        if (!wait(&sb.p_full[u & 3], full_par(u >> 2))) { ok = false; break; }
                        tc_fence_after();
                        // A = dS^T (dK) or P^T (dV): K = 16 query steps at X columns
                        // 0, 8, 32, 40 (dS^T) and 16, 24, 48, 56 (P^T), as the math wrote them
                        const uint64_t xd = tcx::desc_head<64>(xaddr + hf * TILE64);
                        const uint32_t xa = tmem + COL_X + xs * 64 + (dvi ? 16 : 0);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_bf16_ts(d_acc, xa + (ks >> 1) * 32 + (ks & 1) * 8, xd + (uint64_t)(ks * 128), id_acc,
                                            (ks > 0 || g > I.g0 || hf > 0) ? 1u : 0u);
                        mma_commit(&sb.x_empty[xs]);
                        issued = true;
                    }
                    if (!ok) break;
                    // the stage's last products: release it unless the next item of the run uses it
                    if (!keep || g < nx.g0) mma_commit(&sb.st_empty[slot]);
                }
                if (!ok) break;
                mma_commit(&sb.o_full[e & 1]);
            }
            if (issued) {
                uint64_t* dn = dvi ? &sb.done3 : &sb.done2;
                mma_commit(dn);
                mbar_wait(dn, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ math warpgroups
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const int row = 32 * qd + lane;               // key row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const uint64_t sl2 = tcx::f2_pack(a.scale_log2, a.scale_log2);
        const uint64_t sc2 = tcx::f2_pack(a.scale, a.scale);
        Slide sl{-1, -1, 0};
        bool kept = false;
        int u = 0, e = 0;
        bool ok = true;
        for (int item = c0; item < c1 && ok; ++item, ++e) {
            const Item I = decode(a, item);
            Item nx;
            const bool keep = keeps(a, I, item, c1, nx);
            sl.begin(kept, I.strip, I.g0, I.g1);
            kept = keep;
            const int s0 = I.kt * BM;
            const int s = s0 + row;                   // this thread's key
            // queries s .. min(s + W - 1, L - 1) see key s (key rows past L are never stored)
            const int spn = min(a.W - 1, a.L - 1 - s);
            const uint32_t span = spn < 0 ? 0u : static_cast<uint32_t>(spn);
            for (int g = I.g0; g <= I.g1 && ok; ++g) {
                const int p = sl.pos(I.g1, g), slot = p % NSLOT;
                const uint32_t stph = static_cast<uint32_t>(p / NSLOT) & 1u;
                for (int hf = 0; hf < 2; ++hf, ++u) {
                    if ((u & 1) != wg) continue;
                    const int xs = u % NX, ys = u % NY;
                    // own x_full first: its completion implies this stage has landed, so
                    // the stage barrier's phase below is unambiguous
                    if (!wait(&sb.x_full[xs], full_par(u / NX)) || !wait(&sb.st_full[slot], stph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int qb = g * BM + hf * BT;
                    // warpgroup-uniform: do the window edge, the diagonal or the sequence end cross the unit?
                    const bool edge = qb < s0 + BM - 1 || qb + BT - 1 > s0 + a.W - 1 || qb + BT > a.L;
                    const uint8_t* vec = sm + OFF_ST + slot * SLOT + VEC_OFF + hf * BT * 4;
                    const uint64_t* nl = reinterpret_cast<const uint64_t*>(vec);              // pairs
                    const uint64_t* nd = reinterpret_cast<const uint64_t*>(vec + BM * 4);
                    const uint32_t xb = tmem + lane_base + COL_X + xs * 64;
                    const uint32_t yb = tmem + lane_base + COL_Y + ys * 64;
#pragma unroll
                    for (int pc = 0; pc < 2; ++pc) {
                        // queries qb + 32 pc .. + 31 of this key row
                        uint32_t r0[16], r1[16], r2[16], r3[16];
                        tmem_ld_32x32b_x16(xb + 32 * pc, r0);
                        tmem_ld_32x32b_x16(xb + 32 * pc + 16, r1);
                        tmem_ld_32x32b_x16(yb + 32 * pc, r2);
                        tmem_ld_32x32b_x16(yb + 32 * pc + 16, r3);
                        tmem_wait_ld();
                        if (pc == 1) {                               // dP^T fully read: free its slot
                            tc_fence_before();
                            mbar_arrive(&sb.y_empty[ys]);
                        }
                        const int cb = qb + 32 * pc - s;             // column 0 relative to s
                        uint32_t pd[16], pp[16];
                        auto body = [&](bool msk) {
#pragma unroll
                            for (int p2 = 0; p2 < 16; ++p2) {
                                const uint32_t* rs = p2 < 8 ? r0 : r1;
                                const uint32_t* rg = p2 < 8 ? r2 : r3;
                                const int tt = 2 * (p2 & 7);
                                float y0, y1;
                                tcx::f2_unpack(
                                    tcx::ffma2(tcx::f2_pack(__uint_as_float(rs[tt]), __uint_as_float(rs[tt + 1])),
                                               sl2, nl[16 * pc + p2]), y0, y1);
                                float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
                                if (msk) {
                                    p0 = static_cast<uint32_t>(cb + 2 * p2) > span ? 0.f : p0;
                                    p1 = static_cast<uint32_t>(cb + 2 * p2 + 1) > span ? 0.f : p1;
                                }
                                const uint64_t p2v = tcx::f2_pack(p0, p1);
                                const uint64_t gd = tcx::ffma2(
                                    tcx::f2_pack(__uint_as_float(rg[tt]), __uint_as_float(rg[tt + 1])), sc2,
                                    nd[16 * pc + p2]);
                                pd[p2] = tcx::pack_bf16x2(tcx::fmul2(p2v, gd));
                                pp[p2] = tcx::pack_bf16x2(p2v);
                            }
                        };
                        if (edge) body(true);
                        else body(false);
                        // dS^T, then P^T, over the 32 S^T columns just read
                        tmem_st_32x32b_x16(xb + 32 * pc, pd);
                        tmem_st_32x32b_x16(xb + 32 * pc + 16, pp);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&sb.p_full[u & 3]);
                }
            }
            if (!ok) break;
            if ((e & 1) != wg) continue;
            // epilogue: dK and dV rows of key s
            if (!wait(&sb.o_full[wg], full_par(e >> 1))) break;
            tc_fence_after();
            const size_t orow = (((size_t)I.b * a.L + s) * a.H + I.h) * 64;
            uint32_t pkk[32], pkv[32];
            load_row64(tmem + lane_base + COL_ACC, pkk);
            load_row64(tmem + lane_base + COL_ACC + 64, pkv);
            tc_fence_before();
            mbar_arrive(&sb.o_empty);                 // the next item may accumulate now
            if (s < a.L) {
                store_row64(a.dk + orow, pkk);
                store_row64(a.dv + orow, pkv);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}
}  // namespace pb

}  // namespace

// Can consecutive items of a strip keep their shared tiles in a ring of
// `nslot` slots filled and released in load order?  Items i = 0 .. n-1 use tiles
// k0(i) .. k1(i) (both non-decreasing, no gaps between items).
// A new tile k takes the slot of tile k - nslot, which is free once the last
// item that uses k - nslot has passed it; that item must not come after the
// first item that needs k, or the ring would wait on itself.
template <typename Range>
bool slide_safe(int n, int nslot, Range range) {
    int pk0 = 0, pk1 = -1;
    std::vector<int> first, last;
    for (int i = 0; i < n; ++i) {
        int k0, k1;
        range(i, k0, k1);
        if (k1 < k0 || (i > 0 && (k0 < pk0 || k1 < pk1 || k0 > pk1 + 1))) return false;
        for (int k = pk1 + 1; k <= k1; ++k) first.push_back(i);    // first[k]: first item needing k
        last.resize(k1 + 1, i);
        for (int k = k0; k <= k1; ++k) last[k] = i;                // last[k]: last item needing k
        pk0 = k0;
        pk1 = k1;
    }
    for (int k = nslot; k <= pk1; ++k)
        if (last[k - nslot] > first[k]) return false;
    return true;
}

size_t swa_bwd_workspace_bytes(int B, int L, int H) {
    const size_t Lp = ((size_t)L + BM - 1) / BM * BM;
    return 2 * (size_t)B * H * Lp * sizeof(float) + 256;
}

cudaError_t launch_swa_bwd_tc(int B, int L, int H, int W, float attn_scale, const void* q,
                              const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, void* ws, int* status,
                              cudaStream_t st, int* launches) {
    SwaBwdArgs a;
    a.B = B; a.L = L; a.H = H; a.W = W;
    a.Lp = (L + BM - 1) / BM * BM;
    a.nQT = (L + BM - 1) / BM;
    a.nKT = a.nQT;
    a.scale = attn_scale;
    a.scale_log2 = attn_scale * kLog2e;
    a.status = status;
    a.lse = lse;
    a.nlse2T = static_cast<float*>(ws);
    a.ndscT = a.nlse2T + (size_t)B * H * a.Lp;
    a.dq = static_cast<__nv_bfloat16*>(dq);
    a.dk = static_cast<__nv_bfloat16*>(dk);
    a.dv = static_cast<__nv_bfloat16*>(dv);
    const uint64_t cols = (uint64_t)H * 64;
    CUtensorMap q128, do128, o128, k64, v64, k128, v128;
    if (!encode_bf16_seq(&q128, q, B, L, cols, BM) || !encode_bf16_seq(&do128, dout, B, L, cols, BM) ||
        !encode_bf16_seq(&o128, o, B, L, cols, BM) || !encode_bf16_seq(&k64, k, B, L, cols, BT) ||
        !encode_bf16_seq(&v64, v, B, L, cols, BT) || !encode_bf16_seq(&k128, k, B, L, cols, BM) ||
        !encode_bf16_seq(&v128, v, B, L, cols, BM))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e;

    // pass A: items (b, h, query tile), 64-key tiles k0 .. k1 each
    a.n_items = B * H * a.nQT;
    a.slide = slide_safe(a.nQT, pa::NSLOT, [&](int qt, int& k0, int& k1) {
        const int lo = qt * BM - W + 1;
        k0 = (lo < 0 ? 0 : lo) / BT;
        k1 = (qt * BM + BM - 1) / BT;
    }) ? 1 : 0;
    int grid = a.n_items < sms ? a.n_items : sms;
    if ((e = cudaFuncSetAttribute(pa::swa_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  pa::SMEM)) != cudaSuccess)
        return e;
    GCA_LAUNCH("swa_bwd_q_tc", st,
               pa::swa_bwd_q_kernel<<<grid, pa::kThreads, pa::SMEM, st>>>(q128, do128, o128, k64, v64, a));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // pass B: items (b, h, key tile), 128-query stages g0 .. g1 each
    a.n_items = B * H * a.nKT;
    a.slide = slide_safe(a.nKT, pb::NSLOT, [&](int kt, int& g0, int& g1) {
        int last = kt * BM + BM - 1 + W - 1;
        if (last > L - 1) last = L - 1;
        g0 = kt;
        g1 = last / BM;
    }) ? 1 : 0;
    grid = a.n_items < sms ? a.n_items : sms;
    if ((e = cudaFuncSetAttribute(pb::swa_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  pb::SMEM)) != cudaSuccess)
        return e;
    GCA_LAUNCH("swa_bwd_kv_tc", st,
               pb::swa_bwd_kv_kernel<<<grid, pb::kThreads, pb::SMEM, st>>>(q128, do128, k128, v128, a));
    if ((e = cudaGetLastError()) == cudaSuccess) *launches += 2;
    return e;
}

}  // namespace gca
