// attn_swa_tc.cu -- sliding-window causal self-attention on the Blackwell tensor
// cores (bf16, d = 64): the fixed-size window self-attention that a DRT layer
// runs before its GCA module (paper summary section 1: top-k past chunks
// combined with sliding-window self-attention; section 4.1.2: a 512-token
// window; the GCA modules are appended after the attention modules).
//
// Token t of a sequence attends to the keys max(0, t - W + 1) .. t:
//   o_t = sum_s softmax_s(attn_scale q_t . k_s) v_s,  lse_t = ln sum_s exp(...).
//
// Design (one persistent CTA per SM, 12 warps, warp-specialised):
//   item       (batch row, 128-token query tile, head); keys come in tiles of
//              128, so both products are M = 128 MMAs (full rate); for
//              W = 512 an item needs at most 5 key tiles, of which only the
//              first (window edge) and the last (causal diagonal) are masked.
//   warp 0     producer: TMA (3-D maps over [B, L, H*d]: rows outside a
//              sequence read as zeros) of the Q tile (lane 0), each key
//              tile's K (lane 0) and V (lane 1) into a 3-stage and a 7-stage ring:
//              a K stage is free once its S product completes, long before
//              the V stage, which waits for P V.
//   warp 1     S issuer and TMEM owner: S = Q K^T into the item's warpgroup's
//              S buffer (128 columns).
//   warp 2     P V issuer: O += P V into the warpgroup's O accumulator, A = P
//              read from tensor memory.
//   warp 3     idle (completes the first warpgroup, which gives registers
//              to the softmax warpgroups with setmaxnreg).
//   warps 4-11 two softmax warpgroups owning alternate items (the online
//              softmax of a row lives in one thread's registers); producer
//              and issuers walk the two current items' tiles interleaved, so
//              one warpgroup's softmax overlaps the other's products.
// Masking: only the tiles that the window edge or the diagonal crosses are
// masked, in registers, by straight-line selects (no per-chunk branches: the
// unrolled exponential loop relies on interleaving across the whole row).
// Tensor memory: S buffers (2 x 128 columns), O accumulators (2 x 64) and P
// buffers (2 x 64: bf16 pairs in the A operand layout) fill the 512 columns.
// With P out of shared memory the P V products read only V there, the P
// stores leave shared memory alone, and the freed 64 KB deepen the K and V
// rings.  (The P V products stay on one issuing thread: a second issuer,
// spinning on its barriers, costs its SM sub-partition's softmax warps more
// issue slots than it saves.)
// Softmax of one tile: the thread reads its row of S (128 columns) from TMEM
// once and frees the buffer at once, so the next S product overlaps this
// tile's arithmetic; the scaling and the row sum use packed f32x2 arithmetic;
// the first 64 keys' P is formed in registers before the wait for the
// previous P V, then P goes to its TMEM buffer 32 keys per store.
// Online softmax with a stale running max: P = exp2(s' - m) is written
// unnormalised; O (TMEM) and the running sum are rescaled only when a tile's
// max exceeds m by more than 2^8, which keeps every P below 256 and the result
// exact up to rounding.  The rescale reads, scales and writes O in TMEM after
// the previous tile's P V has completed.
// Epilogue: O / l in bf16 goes into the warpgroup's own staging tile in the
// swizzled layout and leaves with one TMA tensor store (rows past the sequence
// end are clipped by the tensor map).  It runs after the next item's first
// row max, so the wait for the last P V overlaps useful work; the store's read
// of the staging tile is awaited only at the following epilogue.
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
using tcx::kLn2;
using tcx::kLog2e;
using tcx::Ring;

constexpr int kThreads = 384;          // control warpgroup + 2 softmax warpgroups
constexpr int kRegsLaunch = 168;       // registers a thread at launch (384 x 168 <= 64K)
constexpr int kRegsCtrl = 56;          // after setmaxnreg: producer / issuer warpgroup
constexpr int kRegsSoftmax = 224;      //                   each softmax warpgroup
static_assert(128 * kRegsCtrl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr int BM = 128;                // query rows per item (MMA M)
constexpr int BN = 128;                // keys per tile (MMA N of S)
constexpr int KST = 3;                 // depth of the K ring (a K stage frees when its S product completes)
constexpr int VST = 7;                 // depth of the V ring (a V stage is held until P V completes)
constexpr int STAGES = KST > VST ? KST : VST;
constexpr int TILE = 128 * 128;        // 128 rows x 64 bf16: a Q, K, V or O tile
constexpr int OFF_Q = 0;               // one Q tile per warpgroup
constexpr int OFF_K = 2 * TILE;
constexpr int OFF_V = OFF_K + KST * TILE;
constexpr int OFF_O = OFF_V + VST * TILE;            // one O staging tile per warpgroup
constexpr int SMEM = OFF_O + 2 * TILE + 1024;           // + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;          // S buffer of warpgroup w at w * 128
constexpr uint32_t COL_O = 256;        // O accumulator of warpgroup w at 256 + w * 64
constexpr uint32_t COL_P = 384;        // P of warpgroup w (bf16 pairs, 128 keys) at 384 + w * 64
constexpr float kRescaleLog2 = 8.f;

struct SwaArgs {
    __nv_bfloat16* o;
    float* lse;              // [B, L, H] or null
    int* status;
    int B, L, H, W, nQT;     // nQT = query tiles per row
    float scale_log2;        // attn_scale * log2(e)
    int n_items;
};

struct __align__(8) Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[STAGES], k_empty[STAGES];
    uint64_t v_full[STAGES], v_empty[STAGES];
    uint64_t epi_full[2], epi_free[2];    // O staged / the previous store has read the staging tile
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t done, done2;
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

// Item -> (batch row, query tile, head), its first key tile and key tile count.
struct Item {
    int b, qt, h, k0, nt;
};
__device__ __forceinline__ Item decode_item(const SwaArgs& a, int item) {
    Item it;
    it.h = item % a.H;
    const int bq = item / a.H;
    it.qt = bq % a.nQT;
    it.b = bq / a.nQT;
    int lo = it.qt * BM - a.W + 1;
    if (lo < 0) lo = 0;
    it.k0 = lo / BN;
    it.nt = it.qt - it.k0 + 1;          // key tiles k0 .. qt (BN == BM)
    return it;
}

// Does key tile j of the item cross the window edge or the diagonal of any of its rows?
__device__ __forceinline__ bool tile_masked(const SwaArgs& a, const Item& it, int j) {
    const int kbase = (it.k0 + j) * BN, t0 = it.qt * BM;
    return kbase + BN - 1 > t0 || kbase < t0 + BM - a.W;
}

__global__ void __launch_bounds__(kThreads, 1)
gca_swa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                      const SwaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ Bars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };
    const int stride = gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.q_full[i], 1);
            mbar_init(&sb.q_empty[i], 1);
            mbar_init(&sb.s_full[i], 1);
            mbar_init(&sb.s_empty[i], 128);
            mbar_init(&sb.p_full[i], 128);
            mbar_init(&sb.p_empty[i], 1);
            mbar_init(&sb.o_full[i], 1);
            mbar_init(&sb.o_empty[i], 128);
        }
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sb.k_full[i], 1);
            mbar_init(&sb.k_empty[i], 1);
            mbar_init(&sb.v_full[i], 1);
            mbar_init(&sb.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.epi_full[i], 128);
            mbar_init(&sb.epi_free[i], 1);
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
        prefetch_tmap(&to);
    }
    if (warp == 1) {
        tmem_alloc(&sb.tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb.tmem;

    // The CTA's items are blockIdx.x + k * gridDim.x; pair p holds k = 2p (warpgroup 0)
    // and k = 2p + 1 (warpgroup 1).  Producer and issuers walk a pair's tiles as
    // (wg 0, tile 0), (wg 1, tile 0), (wg 0, tile 1), ...
    if (warp < 4) {
    // each warpgroup's setmaxnreg heads its own branch: every warp of the group
    // executes that one instruction, and it dominates the code that runs under it
    setmaxnreg_dec<kRegsCtrl>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0: Q tiles and the K ring; lane 1: the V ring (each walks the same
        // sequence of positions and waits on its own barriers)
        if (lane < 2) {
            const bool kl = lane == 0;
            Ring rg{0, 0};
            int kq[2] = {0, 0};
            bool out[STAGES] = {}, q_out[2] = {false, false};
            uint32_t ph[STAGES] = {}, q_ph[2] = {0, 0};
            uint64_t* full = kl ? sb.k_full : sb.v_full;
            uint64_t* empty = kl ? sb.k_empty : sb.v_empty;
            const CUtensorMap* map = kl ? &tk : &tv;
            uint8_t* ring = sm + (kl ? OFF_K : OFF_V);
            const int nst = kl ? KST : VST;
            bool ok = true;
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                Item it[2];
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = 0;
                    if (e < a.n_items) { it[w] = decode_item(a, e); n[w] = it[w].nt; }
                }
                if (kl)
                    for (int w = 0; w < 2 && ok; ++w) {
                        if (n[w] == 0) continue;
                        if (!wait(&sb.q_empty[w], empty_par(kq[w]))) { ok = false; break; }
                        mbar_arrive_expect_tx(&sb.q_full[w], TILE);
                        tma_load_3d(sm + OFF_Q + w * TILE, &tq, &sb.q_full[w], it[w].h * 64,
                                    it[w].qt * BM, it[w].b);
                        q_out[w] = true;
                        q_ph[w] = full_par(kq[w]);
                        ++kq[w];
                    }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if (!wait(&empty[rg.i], rg.ph ^ 1u)) { ok = false; break; }
                        mbar_arrive_expect_tx(&full[rg.i], TILE);
                        tma_load_3d(ring + rg.i * TILE, map, &full[rg.i], it[w].h * 64,
                                    (it[w].k0 + j) * BN, it[w].b);
                        out[rg.i] = true;
                        ph[rg.i] = rg.ph;
                        rg.next(nst);
                    }
            }
            // no copy may still be writing shared memory when the CTA exits
            for (int i = 0; i < nst; ++i)
                if (out[i]) mbar_wait(&full[i], ph[i], nullptr, 100000000ull);
            for (int i = 0; i < 2; ++i)
                if (q_out[i]) mbar_wait(&sb.q_full[i], q_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S issuer
        if (lane == 0) {
            Ring kv{0, 0};
            int kq[2] = {0, 0}, ts[2] = {0, 0};
            bool issued = false, ok = true;
            const uint32_t id_s = idesc_bf16(BM, BN, false, false);
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = e < a.n_items ? decode_item(a, e).nt : 0;
                }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if ((j == 0 && !wait(&sb.q_full[w], full_par(kq[w]))) ||
                            !wait(&sb.k_full[kv.i], kv.ph) ||
                            !wait(&sb.s_empty[w], empty_par(ts[w]))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t qaddr = smem_u32(sm + OFF_Q + w * TILE);
                        const uint32_t kaddr = smem_u32(sm + OFF_K + kv.i * TILE);
                        tcx::mma_kmajor_k64(tmem + COL_S + w * 128, qaddr, kaddr, id_s, 0);
                        mma_commit(&sb.s_full[w]);
                        mma_commit(&sb.k_empty[kv.i]);     // K is read only by this product
                        issued = true;
                        ++ts[w];
                        if (j == n[w] - 1) {
                            mma_commit(&sb.q_empty[w]);    // Q is read only by these products
                            ++kq[w];
                        }
                        kv.next(KST);
                    }
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ P V issuer
        if (lane == 0) {
            Ring kv{0, 0};
            int ko[2] = {0, 0}, tp[2] = {0, 0};
            bool issued = false, ok = true;
            const uint32_t id_o = idesc_bf16(BM, 64, false, true);
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = e < a.n_items ? decode_item(a, e).nt : 0;
                }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if ((j == 0 && !wait(&sb.o_empty[w], empty_par(ko[w]))) ||
                            !wait(&sb.p_full[w], full_par(tp[w])) ||
                            !wait(&sb.v_full[kv.i], kv.ph)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t vaddr = smem_u32(sm + OFF_V + kv.i * TILE);
                        tcx::mma_ts_mn_dh<64, 8>(tmem + COL_O + w * 64, tmem + COL_P + w * 64, vaddr, BN, id_o,
                                                 j > 0);
                        mma_commit(&sb.v_empty[kv.i]);
                        mma_commit(&sb.p_empty[w]);
                        issued = true;
                        ++tp[w];
                        if (j == n[w] - 1) {
                            mma_commit(&sb.o_full[w]);
                            ++ko[w];
                        }
                        kv.next(VST);
                    }
            }
            if (issued) {
                mma_commit(&sb.done2);
                mbar_wait(&sb.done2, 0, nullptr, 100000000ull);
            }
        }
    }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        setmaxnreg_inc<kRegsSoftmax>();
        const int wg = (warp - 4) >> 2;
        const int qd = warp & 3;                        // TMEM lane quarter of this warp
        const int row = 32 * qd + lane;                 // TMEM lane = query row of the tile
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const uint32_t ts_addr = tmem + lane_base + COL_S + wg * 128;
        const uint32_t to_addr = tmem + lane_base + COL_O + wg * 64;
        const uint32_t tp_addr = tmem + lane_base + COL_P + wg * 64;
        uint8_t* const obuf = sm + OFF_O + wg * TILE;
        const bool leader = qd == 0 && lane == 0;       // issues this warpgroup's O stores
        const float sl = a.scale_log2;
        // warp-uniform result: the TMEM accesses and votes after a wait are warp-collective,
        // so a wait that gave up in one lane (abort) must give up in all of them
        auto wwait = [&](uint64_t* bar, uint32_t par) { return __all_sync(0xffffffffu, wait(bar, par)); };

        int ts = 0, ko = 0;
        int item = blockIdx.x + wg * stride, j = 0;
        Item it{};
        if (item < a.n_items) it = decode_item(a, item);
        float m = -INFINITY;                            // running max of s * scale * log2(e)
        float l = 0.f;                                  // running sum of exp2(. - m)
        // the finished item whose O still sits in TMEM
        bool pend = false;
        Item pit{};
        float pm = 0.f, pl = 1.f;
        while (true) {
            const bool have = item < a.n_items;
            float alpha = 1.f;
            bool resc = false;
            float x[128];
            if (have) {
                if (!wwait(&sb.s_full[wg], full_par(ts))) break;
                tc_fence_after();
                float mt;                               // the tile's row max of s
                {
                    // two 64-column loads, each returning its columns' max as well
                    uint32_t r[2][64];
                    float mc[2];
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) mc[ci] = tmem_ld_max_32x32b_x64(ts_addr + 64 * ci, r[ci]);
                    tmem_wait_ld();
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci)
#pragma unroll
                        for (int u = 0; u < 64; ++u) x[64 * ci + u] = __uint_as_float(r[ci][u]);
                    mt = fmaxf(mc[0], mc[1]);
                }
                tc_fence_before();
                mbar_arrive(&sb.s_empty[wg]);           // S is in registers: the buffer is free
                if (tile_masked(a, it, j)) {
                    // row t sees the keys t - W + 1 .. t: columns c_lo .. c_lo + W - 1
                    // (a select per column; a conditional store here becomes a branch);
                    // the max is then taken again over the visible columns
                    const int c_lo = it.qt * BM + row - a.W + 1 - (it.k0 + j) * BN;
                    const uint32_t span = static_cast<uint32_t>(a.W - 1);
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        x[i] = static_cast<uint32_t>(i - c_lo) > span ? -INFINITY : x[i];
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < 128; ++i) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
                    mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                }
                const float mts = mt * sl;
                if (mts > m + kRescaleLog2) {
                    if (m != -INFINITY) {
                        resc = true;
                        alpha = fast_exp2(m - mts);
                    }
                    m = mts;
                }
                l *= alpha;
            }
            // the previous item's output leaves after the next item's first row max,
            // which gives its last P V time to complete
            if ((j == 0 || !have) && pend) {
                if (!wwait(&sb.o_full[wg], full_par(ko))) break;
                tc_fence_after();
                uint32_t r[4][16];
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) tmem_ld_32x32b_x16(to_addr + 16 * ci, r[ci]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sb.o_empty[wg]);
                // the previous store of this warpgroup must have read the staging tile
                if (ko > 0) {
                    if (leader) {
                        bulk_wait_group_read0();
                        mbar_arrive(&sb.epi_free[wg]);
                    }
                    if (!wwait(&sb.epi_free[wg], full_par(ko - 1))) break;
                }
                const float inv = 1.f / pl;
                uint8_t* orow = obuf + row * 128;
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) {
                    float f[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) f[u] = __uint_as_float(r[ci][u]);
                    *reinterpret_cast<uint4*>(orow + (((2 * ci) ^ (row & 7)) << 4)) = tcx::pack8(f, inv);
                    *reinterpret_cast<uint4*>(orow + (((2 * ci + 1) ^ (row & 7)) << 4)) =
                        tcx::pack8(f + 8, inv);
                }
                fence_proxy_async_smem();
                mbar_arrive(&sb.epi_full[wg]);
                const int t = pit.qt * BM + row;
                if (t < a.L && a.lse) a.lse[((size_t)pit.b * a.L + t) * a.H + pit.h] = (pm + log2f(pl)) * kLn2;
                if (leader) {
                    if (!wait(&sb.epi_full[wg], full_par(ko))) break;
                    tma_store_3d(&to, obuf, pit.h * 64, pit.qt * BM, pit.b);
                    bulk_commit_group();
                }
                ++ko;
                pend = false;
            }
            if (!have) break;
            const float mu = (m == -INFINITY) ? 0.f : m;
            const uint64_t sl2 = tcx::f2_pack(sl, sl), nmu2 = tcx::f2_pack(-mu, -mu);
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
            // the first 64 keys' P is formed before the wait for the P buffer
            uint32_t pka[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float y0, y1;
                tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(x[2 * c], x[2 * c + 1]), sl2, nmu2), y0, y1);
                const float e0 = fast_exp2(y0);
                const float e1 = fast_exp2(y1);
                acc2[c & 3] = tcx::fadd2(acc2[c & 3], tcx::f2_pack(e0, e1));
                pka[c] = tcx::pack_bf16(e0, e1);
            }
            // the previous tile's P V has completed: O is stable, P buffer free
            if (!wwait(&sb.p_empty[wg], empty_par(ts))) break;
            if (__any_sync(0xffffffffu, resc)) {
                tc_fence_after();
#pragma unroll 1
                for (int ci = 0; ci < 4; ++ci) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(to_addr + 16 * ci, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 16; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * alpha);
                    tmem_st_32x32b_x16(to_addr + 16 * ci, r);
                }
                tmem_wait_st();
            }
            {                                           // the first 64 keys' P into the buffer
                uint32_t h0[16], h1[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) { h0[u] = pka[u]; h1[u] = pka[16 + u]; }
                tmem_st_32x32b_x16(tp_addr, h0);
                tmem_st_32x32b_x16(tp_addr + 16, h1);
            }
            // p = exp2(s * scale * log2(e) - m) for the other 64 keys; the scaling and the
            // row sum run on column pairs (packed f32x2 FMA and add: one instruction for two)
            uint32_t pk2[16];
#pragma unroll
            for (int c = 4; c < 8; ++c) {
                uint32_t pk[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float y0, y1;
                    const uint64_t s2 = tcx::f2_pack(x[16 * c + 2 * u], x[16 * c + 2 * u + 1]);
                    tcx::f2_unpack(tcx::ffma2(s2, sl2, nmu2), y0, y1);
                    const float e0 = fast_exp2(y0);
                    const float e1 = fast_exp2(y1);
                    acc2[u & 3] = tcx::fadd2(acc2[u & 3], tcx::f2_pack(e0, e1));
                    pk[u] = tcx::pack_bf16(e0, e1);
                }
                if (c & 1) {                            // 16 keys a column pair: store 32 keys
#pragma unroll
                    for (int u = 0; u < 8; ++u) pk2[8 + u] = pk[u];
                    tmem_st_32x32b_x16(tp_addr + 16 * (c >> 1), pk2);
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u) pk2[u] = pk[u];
                }
            }
            tmem_wait_st();
            float l4[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) tcx::f2_unpack(acc2[u], l4[2 * u], l4[2 * u + 1]);
            l += ((l4[0] + l4[1]) + (l4[2] + l4[3])) + ((l4[4] + l4[5]) + (l4[6] + l4[7]));
            tc_fence_before();
            mbar_arrive(&sb.p_full[wg]);
            ++ts;
            if (++j == it.nt) {                         // item done: its O is written out later
                pend = true;
                pit = it;
                pm = m;
                pl = l;
                m = -INFINITY;
                l = 0.f;
                j = 0;
                item += 2 * stride;
                if (item < a.n_items) it = decode_item(a, item);
            }
        }
        // the last tile stores must be complete before the CTA exits
        if (leader) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_swa_fwd_tc(int B, int L, int H, int W, float attn_scale, const void* q,
                              const void* k, const void* v, void* o, float* lse, int* status,
                              cudaStream_t st, int* launches) {
    CUtensorMap tq, tk, tv, to;
    const uint64_t cols = (uint64_t)H * 64;
    if (!encode_bf16_seq(&tq, q, B, L, cols, BM) || !encode_bf16_seq(&tk, k, B, L, cols, BN) ||
        !encode_bf16_seq(&tv, v, B, L, cols, BN) || !encode_bf16_seq(&to, o, B, L, cols, BM))
        return cudaErrorInvalidValue;
    SwaArgs a;
    a.o = static_cast<__nv_bfloat16*>(o);
    a.lse = lse;
    a.status = status;
    a.B = B; a.L = L; a.H = H; a.W = W;
    a.nQT = (L + BM - 1) / BM;
    a.scale_log2 = attn_scale * kLog2e;
    a.n_items = B * a.nQT * H;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = a.n_items < sms ? a.n_items : sms;
    // the setmaxnreg split needs the whole launch allocation: refuse to launch a
    // build that gave the kernel fewer registers a thread (its warps would wait forever)
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, gca_swa_fwd_tc_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < 128 * kRegsCtrl + 256 * kRegsSoftmax) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(gca_swa_fwd_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    GCA_LAUNCH("swa_fwd_tc", st, gca_swa_fwd_tc_kernel<<<grid, kThreads, SMEM, st>>>(tq, tk, tv, to, a));
    if ((e = cudaGetLastError()) == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace gca
