// attn_swa_bwd_tc.cu -- backward of the sliding-window causal self-attention
// (the 512-token window self-attention a DRT layer runs before its GCA
// module; paper summary sections 1 and 4.1.2) on the Blackwell tensor cores
// (bf16, d = 64).
//
// With p_ts = exp(attn_scale q_t . k_s - lse_t) over the window of t,
// delta_t = dO_t . O_t, dp_ts = dO_t . v_s and ds_ts = attn_scale p_ts (dp_ts - delta_t):
//   dQ_t = sum_s ds_ts k_s,   dK_s = sum_t ds_ts q_t,   dV_s = sum_t p_ts dO_t.
// Three launches, no atomics (every output row is written by one CTA):
//   swa_delta    delta and lse * log2(e) per (token, head), stored as [B, H, Lp]
//                rows so that 64 consecutive tokens are one bulk copy.
//   pass A       query-major, item = (batch row, 128-token query tile, head):
//                for each 64-key tile S = Q K^T and dP = dO V^T (M = 128,
//                N = 64) into the warpgroup's TMEM buffer, ds in registers,
//                dQ += dS K accumulated in TMEM.
//   pass B       key-major, item = (batch row, 128-key tile, head): for each
//                64-query tile S^T = K Q^T and dP^T = V dO^T, then
//                dV += P^T dO and dK += dS^T Q accumulated in TMEM.
// Warp roles as in the forward: warp 0 producer (lane 0 and lane 1 feed two
// rings), warp 1 score-product issuer and TMEM owner, warp 2 accumulation
// issuer, warps 3-10 two math warpgroups owning alternate items; producer and
// issuers walk the two current items' tiles interleaved.  Outputs are staged
// in the warpgroup's idle operand buffer and written with TMA tensor stores
// (3-D maps over [B, L, H*d]: rows past a sequence end are read as zeros and
// never written).  Every mbarrier wait is bounded.
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
using tcx::Ring;

constexpr int kThreads = 352;
constexpr int BM = 128;                  // item rows = MMA M
constexpr int BT = 64;                   // inner tile = MMA N of the score products
constexpr int STAGES = 4;
constexpr int TILE128 = 128 * 128;       // 128 rows x 64 bf16
constexpr int TILE64 = 64 * 128;         // 64 rows x 64 bf16
constexpr int OPB = BM * 128;            // one operand buffer: 128 rows x 64 bf16
constexpr uint32_t TMEM_COLS = 512;

struct SwaBwdArgs {
    const float* lse2T;      // [B, H, Lp]: lse * log2(e)
    const float* deltaT;     // [B, H, Lp]
    int* status;
    int B, L, H, W, Lp;
    int nQT, nKT, nQ64;      // 128-token query tiles, 128-key tiles, 64-token query tiles per row
    float scale_log2;        // attn_scale * log2(e)
    float scale;             // attn_scale
    int n_items;
};

__device__ __forceinline__ uint32_t full_par(int k) { return static_cast<uint32_t>(k) & 1u; }
__device__ __forceinline__ uint32_t empty_par(int k) { return (static_cast<uint32_t>(k) & 1u) ^ 1u; }

// ---------------------------------------------------------------- delta
__global__ void swa_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                 const __nv_bfloat16* __restrict__ dout,
                                 const float* __restrict__ lse, int B, int L, int H, int Lp,
                                 float* __restrict__ lse2T, float* __restrict__ deltaT) {
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)B * H * Lp;
    if (idx >= total) return;
    const int t = (int)(idx % Lp);
    const size_t bh = idx / Lp;
    const int h = (int)(bh % H), b = (int)(bh / H);
    float dl = 0.f, l2 = 0.f;
    if (t < L) {
        const size_t row = ((size_t)b * L + t) * H + h;
        const uint4* po = reinterpret_cast<const uint4*>(o + row * 64);
        const uint4* pg = reinterpret_cast<const uint4*>(dout + row * 64);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const uint4 a = __ldg(po + v), g = __ldg(pg + v);
            const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* hg = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 fa = __bfloat1622float2(ha[u]), fg = __bfloat1622float2(hg[u]);
                acc[2 * u] = fmaf(fa.x, fg.x, acc[2 * u]);
                acc[2 * u + 1] = fmaf(fa.y, fg.y, acc[2 * u + 1]);
            }
        }
        dl = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        l2 = lse[row] * kLog2e;
    }
    deltaT[idx] = dl;
    lse2T[idx] = l2;
}

// Row of `x` (64 fp32 values of one thread) -> bf16 into a swizzled 128-row x
// 64-column operand tile (row r at r * 128 bytes, 16-byte chunk c at c ^ (r & 7)).
__device__ __forceinline__ void put_row64(uint8_t* buf, int row, const uint32_t (&pk)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(buf + row * 128 + ((c ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}

// 64 TMEM columns of this thread's lane -> fp32 registers.
__device__ __forceinline__ void load64(uint32_t taddr, float (&x)[64]) {
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr + 16 * ci, r);
#pragma unroll
        for (int u = 0; u < 16; ++u) x[16 * ci + u] = __uint_as_float(r[u]);
    }
}

// ============================================================================ pass A (dQ)
namespace pa {
constexpr int OFF_QD = 0;                        // per warpgroup: Q tile, dO tile
constexpr int OFF_K = 2 * 2 * TILE128;
constexpr int OFF_V = OFF_K + STAGES * TILE64;
constexpr int OFF_DS = OFF_V + STAGES * TILE64;  // per warpgroup: dS operand (and dQ staging)
constexpr int SMEM = OFF_DS + 2 * OPB + 1024;
constexpr uint32_t COL_S = 0;                    // warpgroup w: S at w*128, dP at w*128 + 64
constexpr uint32_t COL_DQ = 256;                 // warpgroup w: dQ at 256 + w*64

struct Item {
    int b, qt, h, k0, nt;    // key tiles of 64: k0 .. k0 + nt - 1
};
__device__ __forceinline__ Item decode(const SwaBwdArgs& a, int item) {
    Item it;
    it.h = item % a.H;
    const int bq = item / a.H;
    it.qt = bq % a.nQT;
    it.b = bq / a.nQT;
    int lo = it.qt * BM - a.W + 1;
    if (lo < 0) lo = 0;
    it.k0 = lo / BT;
    it.nt = (it.qt * BM + BM - 1) / BT - it.k0 + 1;
    return it;
}

struct __align__(8) Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
    uint64_t s_full[2], s_empty[2];
    uint64_t ds_full[2], ds_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t epi_full[2], epi_free[2];
    uint64_t done, done2;
    uint32_t tmem;
    int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
swa_bwd_q_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                 const __grid_constant__ CUtensorMap tdq, const SwaBwdArgs a) {
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
            mbar_init(&sb.ds_full[i], 128);
            mbar_init(&sb.ds_empty[i], 1);
            mbar_init(&sb.o_full[i], 1);
            mbar_init(&sb.o_empty[i], 128);
            mbar_init(&sb.epi_full[i], 128);
            mbar_init(&sb.epi_free[i], 1);
        }
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sb.k_full[i], 1);
            mbar_init(&sb.k_empty[i], 1);
            mbar_init(&sb.v_full[i], 1);
            mbar_init(&sb.v_empty[i], 1);
        }
        mbar_init(&sb.done, 1);
        mbar_init(&sb.done2, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tdo);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tdq);
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
        // lane 0: Q / dO tiles and the K ring; lane 1: the V ring
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
            bool ok = true;
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                Item it[2];
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = 0;
                    if (e < a.n_items) { it[w] = decode(a, e); n[w] = it[w].nt; }
                }
                if (kl)
                    for (int w = 0; w < 2 && ok; ++w) {
                        if (n[w] == 0) continue;
                        if (!wait(&sb.q_empty[w], empty_par(kq[w]))) { ok = false; break; }
                        uint8_t* qb = sm + OFF_QD + w * 2 * TILE128;
                        mbar_arrive_expect_tx(&sb.q_full[w], 2 * TILE128);
                        tma_load_3d(qb, &tq, &sb.q_full[w], it[w].h * 64, it[w].qt * BM, it[w].b);
                        tma_load_3d(qb + TILE128, &tdo, &sb.q_full[w], it[w].h * 64, it[w].qt * BM, it[w].b);
                        q_out[w] = true;
                        q_ph[w] = full_par(kq[w]);
                        ++kq[w];
                    }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if (!wait(&empty[rg.i], rg.ph ^ 1u)) { ok = false; break; }
                        mbar_arrive_expect_tx(&full[rg.i], TILE64);
                        tma_load_3d(ring + rg.i * TILE64, map, &full[rg.i], it[w].h * 64,
                                    (it[w].k0 + j) * BT, it[w].b);
                        out[rg.i] = true;
                        ph[rg.i] = rg.ph;
                        rg.next(STAGES);
                    }
            }
            for (int i = 0; i < STAGES; ++i)
                if (out[i]) mbar_wait(&full[i], ph[i], nullptr, 100000000ull);
            for (int i = 0; i < 2; ++i)
                if (q_out[i]) mbar_wait(&sb.q_full[i], q_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S / dP issuer
        if (lane == 0) {
            Ring rg{0, 0};
            int kq[2] = {0, 0}, ts[2] = {0, 0};
            bool issued = false, ok = true;
            const uint32_t id_s = idesc_bf16(BM, BT, false, false);
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = e < a.n_items ? decode(a, e).nt : 0;
                }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if ((j == 0 && !wait(&sb.q_full[w], full_par(kq[w]))) ||
                            !wait(&sb.k_full[rg.i], rg.ph) || !wait(&sb.v_full[rg.i], rg.ph) ||
                            !wait(&sb.s_empty[w], empty_par(ts[w]))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t qaddr = smem_u32(sm + OFF_QD + w * 2 * TILE128);
                        const uint32_t kaddr = smem_u32(sm + OFF_K + rg.i * TILE64);
                        const uint32_t vaddr = smem_u32(sm + OFF_V + rg.i * TILE64);
                        tcx::mma_kmajor_k64(tmem + COL_S + w * 128, qaddr, kaddr, id_s, 0);
                        tcx::mma_kmajor_k64(tmem + COL_S + w * 128 + BT, qaddr + TILE128, vaddr, id_s, 0);
                        mma_commit(&sb.s_full[w]);
                        mma_commit(&sb.v_empty[rg.i]);        // V is read only by dP
                        issued = true;
                        ++ts[w];
                        if (j == n[w] - 1) {
                            mma_commit(&sb.q_empty[w]);       // Q and dO are read only here
                            ++kq[w];
                        }
                        rg.next(STAGES);
                    }
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ dQ issuer
        if (lane == 0) {
            Ring rg{0, 0};
            int ko[2] = {0, 0}, td[2] = {0, 0};
            bool issued = false, ok = true;
            const uint32_t id_dq = idesc_bf16(BM, 64, false, true);
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = e < a.n_items ? decode(a, e).nt : 0;
                }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if ((j == 0 && !wait(&sb.o_empty[w], empty_par(ko[w]))) ||
                            !wait(&sb.ds_full[w], full_par(td[w]))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t dsaddr = smem_u32(sm + OFF_DS + w * OPB);
                        const uint32_t kaddr = smem_u32(sm + OFF_K + rg.i * TILE64);
                        tcx::mma_kmajor_mnmajor<4>(tmem + COL_DQ + w * 64, dsaddr, OPB, kaddr, id_dq, j > 0);
                        mma_commit(&sb.k_empty[rg.i]);
                        mma_commit(&sb.ds_empty[w]);
                        issued = true;
                        ++td[w];
                        if (j == n[w] - 1) {
                            mma_commit(&sb.o_full[w]);
                            ++ko[w];
                        }
                        rg.next(STAGES);
                    }
            }
            if (issued) {
                mma_commit(&sb.done2);
                mbar_wait(&sb.done2, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ math warpgroups
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const uint32_t ts_addr = tmem + lane_base + COL_S + wg * 128;
        const uint32_t tq_addr = tmem + lane_base + COL_DQ + wg * 64;
        uint8_t* dsbuf = sm + OFF_DS + wg * OPB;
        int ts = 0, ko = 0;
        bool ok = true;
        for (int item = blockIdx.x + wg * stride; item < a.n_items && ok; item += 2 * stride) {
            const Item it = decode(a, item);
            const int t0 = it.qt * BM;
            const int t = t0 + row;
            const size_t vrow = ((size_t)it.b * a.H + it.h) * a.Lp + t;   // t < Lp
            const float lse2 = a.lse2T[vrow];
            const float dlt = a.deltaT[vrow];
            const uint64_t nsl2 = tcx::f2_pack(-a.scale_log2, -a.scale_log2), l2 = tcx::f2_pack(lse2, lse2);
            const uint64_t sc2 = tcx::f2_pack(a.scale, a.scale);
            const uint64_t ndsc2 = tcx::f2_pack(-dlt * a.scale, -dlt * a.scale);
            const uint32_t span = static_cast<uint32_t>(a.W - 1);
            for (int j = 0; j < it.nt; ++j) {
                if (!wait(&sb.s_full[wg], full_par(ts))) { ok = false; break; }
                tc_fence_after();
                const int kbase = (it.k0 + j) * BT;
                const bool edge = kbase + BT - 1 > t0 || kbase < t0 + BM - a.W;
                const int lo = t - a.W + 1;
                // the previous dQ product has read the dS buffer (for a first tile: the
                // previous item's dQ store has read it too)
                if (!wait(&sb.ds_empty[wg], empty_par(ts)) ||
                    (j == 0 && ko > 0 && !wait(&sb.epi_free[wg], full_par(ko - 1)))) { ok = false; break; }
                // 32 columns at a time: S and dP from TMEM, dS out 8 columns (16 bytes) at a time
                for (int hf = 0; hf < 2; ++hf) {
                    float x[32], g[32];
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) {
                        uint32_t r[16], q[16];
                        tmem_ld_32x32b_x16(ts_addr + 32 * hf + 16 * ci, r);
                        tmem_ld_32x32b_x16(ts_addr + BT + 32 * hf + 16 * ci, q);
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            x[16 * ci + u] = __uint_as_float(r[u]);
                            g[16 * ci + u] = __uint_as_float(q[u]);
                        }
                    }
                    tmem_wait_ld();
                    if (hf == 1) {                      // S and dP fully read
                        tc_fence_before();
                        mbar_arrive(&sb.s_empty[wg]);
                    }
                    // column pairs in packed f32x2 arithmetic: p = exp2(-(lse2 - s sl)),
                    // dS = p (dP - delta) scale; on a tile that the window edge or the
                    // diagonal crosses, key t0 + c outside [lo, t] gets p = 0 (a select)
                    uint32_t pk[16];
                    const int cb = kbase + 32 * hf - lo;          // column 0 relative to lo
                    auto body = [&](bool msk) {
#pragma unroll
                        for (int pi = 0; pi < 16; ++pi) {
                            float y0, y1;
                            tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(x[2 * pi], x[2 * pi + 1]), nsl2, l2), y0, y1);
                            float p0 = fast_exp2(-y0), p1 = fast_exp2(-y1);
                            if (msk) {
                                p0 = static_cast<uint32_t>(cb + 2 * pi) > span ? 0.f : p0;
                                p1 = static_cast<uint32_t>(cb + 2 * pi + 1) > span ? 0.f : p1;
                            }
                            const uint64_t gd = tcx::ffma2(tcx::f2_pack(g[2 * pi], g[2 * pi + 1]), sc2, ndsc2);
                            pk[pi] = tcx::pack_bf16x2(tcx::fmul2(tcx::f2_pack(p0, p1), gd));
                        }
                    };
                    if (edge) body(true);
                    else body(false);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const int chunk = 4 * hf + ch;
                        *reinterpret_cast<uint4*>(dsbuf + row * 128 + ((chunk ^ (row & 7)) << 4)) =
                            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&sb.ds_full[wg]);
                ++ts;
            }
            if (!ok) break;
            // epilogue: dQ (TMEM) -> bf16 rows in the idle dS buffer -> one tensor store
            if (!wait(&sb.o_full[wg], full_par(ko))) break;
            tc_fence_after();
            float x[64];
            load64(tq_addr, x);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&sb.o_empty[wg]);
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) pk[i] = tcx::pack_bf16(x[2 * i], x[2 * i + 1]);
            put_row64(dsbuf, row, pk);
            fence_proxy_async_smem();
            mbar_arrive(&sb.epi_full[wg]);
            if (qd == 0 && lane == 0) {
                if (!wait(&sb.epi_full[wg], full_par(ko))) break;
                tma_store_3d(&tdq, dsbuf, it.h * 64, t0, it.b);
                bulk_commit_group();
                bulk_wait_group_read0();
                mbar_arrive(&sb.epi_free[wg]);
            }
            ++ko;
        }
        if (qd == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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
constexpr int OFF_KV = 0;                        // per warpgroup: K tile, V tile
constexpr int VEC = TILE64;                      // 64 fp32 after each Q / dO tile (lse2 / delta)
constexpr int STAGE = TILE64 + 1024;
constexpr int OFF_Q = 2 * 2 * TILE128;
constexpr int OFF_DO = OFF_Q + STAGES * STAGE;
constexpr int OFF_OP = OFF_DO + STAGES * STAGE;  // per warpgroup: P^T operand, dS^T operand
constexpr int SMEM = OFF_OP + 2 * 2 * OPB + 1024;
constexpr uint32_t COL_S = 0;                    // warpgroup w: S^T at w*128, dP^T at w*128 + 64
constexpr uint32_t COL_ACC = 256;                // warpgroup w: dK at 256 + w*128, dV at +64

struct Item {
    int b, kt, h, q0, nt;    // query tiles of 64: q0 .. q0 + nt - 1
};
__device__ __forceinline__ Item decode(const SwaBwdArgs& a, int item) {
    Item it;
    it.h = item % a.H;
    const int bk = item / a.H;
    it.kt = bk % a.nKT;
    it.b = bk / a.nKT;
    it.q0 = it.kt * BM / BT;
    int hi = (it.kt * BM + BM - 1 + a.W - 1) / BT;
    if (hi > a.nQ64 - 1) hi = a.nQ64 - 1;
    it.nt = hi - it.q0 + 1;
    return it;
}

struct __align__(8) Bars {
    uint64_t kv_full[2], kv_empty[2];
    uint64_t q_full[STAGES], q_empty[STAGES], d_full[STAGES], d_empty[STAGES];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t epi_full[2], epi_free[2];
    uint64_t done, done2;
    uint32_t tmem;
    int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
swa_bwd_kv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                  const SwaBwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ Bars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto wait = [&](uint64_t* bar, uint32_t par) { return tcx::wait_bar(&sb.abort, bar, par, a.status); };
    const int stride = gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sb.kv_full[i], 1);
            mbar_init(&sb.kv_empty[i], 1);
            mbar_init(&sb.s_full[i], 1);
            mbar_init(&sb.s_empty[i], 128);
            mbar_init(&sb.p_full[i], 128);
            mbar_init(&sb.p_empty[i], 1);
            mbar_init(&sb.o_full[i], 1);
            mbar_init(&sb.o_empty[i], 128);
            mbar_init(&sb.epi_full[i], 128);
            mbar_init(&sb.epi_free[i], 1);
        }
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sb.q_full[i], 1);
            mbar_init(&sb.q_empty[i], 1);
            mbar_init(&sb.d_full[i], 1);
            mbar_init(&sb.d_empty[i], 1);
        }
        mbar_init(&sb.done, 1);
        mbar_init(&sb.done2, 1);
        sb.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tdo);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tdk);
        prefetch_tmap(&tdv);
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
        // lane 0: K / V tiles and the Q ring (+ lse2 rows); lane 1: the dO ring (+ delta rows)
        if (lane < 2) {
            const bool ql = lane == 0;
            Ring rg{0, 0};
            int kk[2] = {0, 0};
            bool out[STAGES] = {}, kv_out[2] = {false, false};
            uint32_t ph[STAGES] = {}, kv_ph[2] = {0, 0};
            uint64_t* full = ql ? sb.q_full : sb.d_full;
            uint64_t* empty = ql ? sb.q_empty : sb.d_empty;
            const CUtensorMap* map = ql ? &tq : &tdo;
            const float* vec = ql ? a.lse2T : a.deltaT;
            uint8_t* ring = sm + (ql ? OFF_Q : OFF_DO);
            bool ok = true;
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                Item it[2];
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = 0;
                    if (e < a.n_items) { it[w] = decode(a, e); n[w] = it[w].nt; }
                }
                if (ql)
                    for (int w = 0; w < 2 && ok; ++w) {
                        if (n[w] == 0) continue;
                        if (!wait(&sb.kv_empty[w], empty_par(kk[w]))) { ok = false; break; }
                        uint8_t* kb = sm + OFF_KV + w * 2 * TILE128;
                        mbar_arrive_expect_tx(&sb.kv_full[w], 2 * TILE128);
                        tma_load_3d(kb, &tk, &sb.kv_full[w], it[w].h * 64, it[w].kt * BM, it[w].b);
                        tma_load_3d(kb + TILE128, &tv, &sb.kv_full[w], it[w].h * 64, it[w].kt * BM, it[w].b);
                        kv_out[w] = true;
                        kv_ph[w] = full_par(kk[w]);
                        ++kk[w];
                    }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if (!wait(&empty[rg.i], rg.ph ^ 1u)) { ok = false; break; }
                        uint8_t* stg = ring + rg.i * STAGE;
                        const int qb = (it[w].q0 + j) * BT;
                        mbar_arrive_expect_tx(&full[rg.i], TILE64 + BT * 4);
                        tma_load_3d(stg, map, &full[rg.i], it[w].h * 64, qb, it[w].b);
                        tcx::bulk_load(stg + VEC, vec + ((size_t)it[w].b * a.H + it[w].h) * a.Lp + qb,
                                       BT * 4, &full[rg.i]);
                        out[rg.i] = true;
                        ph[rg.i] = rg.ph;
                        rg.next(STAGES);
                    }
            }
            for (int i = 0; i < STAGES; ++i)
                if (out[i]) mbar_wait(&full[i], ph[i], nullptr, 100000000ull);
            for (int i = 0; i < 2; ++i)
                if (kv_out[i]) mbar_wait(&sb.kv_full[i], kv_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S^T / dP^T issuer
        if (lane == 0) {
            Ring rg{0, 0};
            int kk[2] = {0, 0}, ts[2] = {0, 0};
            bool issued = false, ok = true;
            const uint32_t id_s = idesc_bf16(BM, BT, false, false);
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = e < a.n_items ? decode(a, e).nt : 0;
                }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if ((j == 0 && !wait(&sb.kv_full[w], full_par(kk[w]))) ||
                            !wait(&sb.q_full[rg.i], rg.ph) || !wait(&sb.d_full[rg.i], rg.ph) ||
                            !wait(&sb.s_empty[w], empty_par(ts[w]))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t kaddr = smem_u32(sm + OFF_KV + w * 2 * TILE128);
                        const uint32_t qaddr = smem_u32(sm + OFF_Q + rg.i * STAGE);
                        const uint32_t daddr = smem_u32(sm + OFF_DO + rg.i * STAGE);
                        tcx::mma_kmajor_k64(tmem + COL_S + w * 128, kaddr, qaddr, id_s, 0);
                        tcx::mma_kmajor_k64(tmem + COL_S + w * 128 + BT, kaddr + TILE128, daddr, id_s, 0);
                        mma_commit(&sb.s_full[w]);
                        issued = true;
                        ++ts[w];
                        if (j == n[w] - 1) {
                            mma_commit(&sb.kv_empty[w]);      // K and V are read only here
                            ++kk[w];
                        }
                        rg.next(STAGES);
                    }
            }
            if (issued) {
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ dK / dV issuer
        if (lane == 0) {
            Ring rg{0, 0};
            int ko[2] = {0, 0}, tp[2] = {0, 0};
            bool issued = false, ok = true;
            const uint32_t id_acc = idesc_bf16(BM, 64, false, true);
            for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
                int n[2];
                for (int w = 0; w < 2; ++w) {
                    const int e = e0 + w * stride;
                    n[w] = e < a.n_items ? decode(a, e).nt : 0;
                }
                const int nmax = n[0] > n[1] ? n[0] : n[1];
                for (int j = 0; j < nmax && ok; ++j)
                    for (int w = 0; w < 2; ++w) {
                        if (j >= n[w]) continue;
                        if ((j == 0 && !wait(&sb.o_empty[w], empty_par(ko[w]))) ||
                            !wait(&sb.p_full[w], full_par(tp[w]))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ptaddr = smem_u32(sm + OFF_OP + w * 2 * OPB);
                        const uint32_t qaddr = smem_u32(sm + OFF_Q + rg.i * STAGE);
                        const uint32_t daddr = smem_u32(sm + OFF_DO + rg.i * STAGE);
                        const uint32_t acc = tmem + COL_ACC + w * 128;
                        tcx::mma_kmajor_mnmajor<4>(acc + 64, ptaddr, OPB, daddr, id_acc, j > 0);        // dV
                        tcx::mma_kmajor_mnmajor<4>(acc, ptaddr + OPB, OPB, qaddr, id_acc, j > 0);       // dK
                        mma_commit(&sb.q_empty[rg.i]);
                        mma_commit(&sb.d_empty[rg.i]);
                        mma_commit(&sb.p_empty[w]);
                        issued = true;
                        ++tp[w];
                        if (j == n[w] - 1) {
                            mma_commit(&sb.o_full[w]);
                            ++ko[w];
                        }
                        rg.next(STAGES);
                    }
            }
            if (issued) {
                mma_commit(&sb.done2);
                mbar_wait(&sb.done2, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ math warpgroups
        const int wg = (warp - 3) >> 2;
        const int qd = warp & 3;
        const int row = 32 * qd + lane;               // key row of the item's tile
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const uint32_t ts_addr = tmem + lane_base + COL_S + wg * 128;
        const uint32_t ta_addr = tmem + lane_base + COL_ACC + wg * 128;
        uint8_t* ptbuf = sm + OFF_OP + wg * 2 * OPB;
        uint8_t* dsbuf = ptbuf + OPB;
        Ring rg{0, 0};
        int ts = 0, ko = 0;
        bool ok = true;
        for (int e0 = blockIdx.x; e0 < a.n_items && ok; e0 += 2 * stride) {
            int n[2];
            Item mine;
            for (int w = 0; w < 2; ++w) {
                const int e = e0 + w * stride;
                n[w] = 0;
                if (e < a.n_items) {
                    const Item it = decode(a, e);
                    n[w] = it.nt;
                    if (w == wg) mine = it;
                }
            }
            if (n[wg] == 0) break;                    // no more items for this warpgroup
            const int s = mine.kt * BM + row;         // this thread's key
            const uint64_t nsl2 = tcx::f2_pack(-a.scale_log2, -a.scale_log2);
            const uint64_t sc2 = tcx::f2_pack(a.scale, a.scale);
            // queries s .. min(s + W - 1, L - 1) see this key (rows past L are never stored)
            const uint32_t span = static_cast<uint32_t>(min(a.W - 1, a.L - 1 - s));
            const int nmax = n[0] > n[1] ? n[0] : n[1];
            for (int j = 0; j < nmax && ok; ++j)
                for (int w = 0; w < 2; ++w) {
                    if (j >= n[w]) continue;
                    const int stg = rg.i;
                    const uint32_t stph = rg.ph;
                    rg.next(STAGES);
                    if (w != wg) continue;
                    if (!wait(&sb.s_full[wg], full_par(ts)) || !wait(&sb.q_full[stg], stph) ||
                        !wait(&sb.d_full[stg], stph)) { ok = false; break; }
                    tc_fence_after();
                    const float4* l4 = reinterpret_cast<const float4*>(sm + OFF_Q + stg * STAGE + VEC);
                    const float4* d4 = reinterpret_cast<const float4*>(sm + OFF_DO + stg * STAGE + VEC);
                    const int qb = (mine.q0 + j) * BT;
                    // warp-uniform: the selects below are exact per lane
                    const bool edge = __any_sync(0xffffffffu, qb < s || qb + BT - 1 > s + a.W - 1 || qb + BT > a.L);
                    // the previous accumulation products have read the operand buffers
                    // (for a first tile: the previous item's stores have read them too)
                    if (!wait(&sb.p_empty[wg], empty_par(ts)) ||
                        (j == 0 && ko > 0 && !wait(&sb.epi_free[wg], full_par(ko - 1)))) { ok = false; break; }
                    // 32 columns at a time: S^T and dP^T from TMEM, P^T and dS^T out to the
                    // operand buffers 8 columns (16 bytes) at a time
                    for (int hf = 0; hf < 2; ++hf) {
                        float x[32], g[32];
#pragma unroll
                        for (int ci = 0; ci < 2; ++ci) {
                            uint32_t r[16], q[16];
                            tmem_ld_32x32b_x16(ts_addr + 32 * hf + 16 * ci, r);
                            tmem_ld_32x32b_x16(ts_addr + BT + 32 * hf + 16 * ci, q);
#pragma unroll
                            for (int u = 0; u < 16; ++u) {
                                x[16 * ci + u] = __uint_as_float(r[u]);
                                g[16 * ci + u] = __uint_as_float(q[u]);
                            }
                        }
                        tmem_wait_ld();
                        if (hf == 1) {                  // S^T and dP^T fully read
                            tc_fence_before();
                            mbar_arrive(&sb.s_empty[wg]);
                        }
                        // query pairs in packed f32x2 arithmetic: P^T = exp2(-(lse2 - s sl)),
                        // dS^T = p (dP - delta) scale; on a tile that the window edges cross,
                        // query tq outside [s, min(s + W - 1, L - 1)] gets p = 0 (a select)
                        const ulonglong2* l2v = reinterpret_cast<const ulonglong2*>(l4) + 8 * hf;
                        const ulonglong2* d2v = reinterpret_cast<const ulonglong2*>(d4) + 8 * hf;
                        const int cb = qb + 32 * hf - s;            // column 0 relative to s
                        uint32_t pp[16], pd[16];
                        auto body = [&](bool msk) {
#pragma unroll
                            for (int pi = 0; pi < 16; ++pi) {
                                const ulonglong2 lv = l2v[pi >> 1], dv = d2v[pi >> 1];
                                float y0, y1;
                                tcx::f2_unpack(tcx::ffma2(tcx::f2_pack(x[2 * pi], x[2 * pi + 1]), nsl2,
                                                          (pi & 1) ? lv.y : lv.x), y0, y1);
                                float p0 = fast_exp2(-y0), p1 = fast_exp2(-y1);
                                if (msk) {
                                    p0 = static_cast<uint32_t>(cb + 2 * pi) > span ? 0.f : p0;
                                    p1 = static_cast<uint32_t>(cb + 2 * pi + 1) > span ? 0.f : p1;
                                }
                                const uint64_t p2 = tcx::f2_pack(p0, p1);
                                const uint64_t g2 = tcx::f2_pack(g[2 * pi], g[2 * pi + 1]);
                                pp[pi] = tcx::pack_bf16x2(p2);
                                pd[pi] = tcx::pack_bf16x2(
                                    tcx::fmul2(tcx::fmul2(p2, sc2), tcx::fsub2(g2, (pi & 1) ? dv.y : dv.x)));
                            }
                        };
                        if (edge) body(true);
                        else body(false);
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            const int chunk = 4 * hf + ch;
                            const int off = row * 128 + ((chunk ^ (row & 7)) << 4);
                            *reinterpret_cast<uint4*>(ptbuf + off) =
                                make_uint4(pp[4 * ch], pp[4 * ch + 1], pp[4 * ch + 2], pp[4 * ch + 3]);
                            *reinterpret_cast<uint4*>(dsbuf + off) =
                                make_uint4(pd[4 * ch], pd[4 * ch + 1], pd[4 * ch + 2], pd[4 * ch + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&sb.p_full[wg]);
                    ++ts;
                }
            if (!ok) break;
            // epilogue: dK, dV (TMEM) -> bf16 rows in the idle operand buffers -> tensor stores
            if (!wait(&sb.o_full[wg], full_par(ko))) break;
            tc_fence_after();
            {
                float x[64];
                uint32_t pk[32];
                load64(ta_addr, x);                   // dK
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = tcx::pack_bf16(x[2 * i], x[2 * i + 1]);
                put_row64(dsbuf, row, pk);
                load64(ta_addr + 64, x);              // dV
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = tcx::pack_bf16(x[2 * i], x[2 * i + 1]);
                put_row64(ptbuf, row, pk);
            }
            tc_fence_before();
            mbar_arrive(&sb.o_empty[wg]);
            fence_proxy_async_smem();
            mbar_arrive(&sb.epi_full[wg]);
            if (qd == 0 && lane == 0) {
                if (!wait(&sb.epi_full[wg], full_par(ko))) break;
                tma_store_3d(&tdk, dsbuf, mine.h * 64, mine.kt * BM, mine.b);
                tma_store_3d(&tdv, ptbuf, mine.h * 64, mine.kt * BM, mine.b);
                bulk_commit_group();
                bulk_wait_group_read0();
                mbar_arrive(&sb.epi_free[wg]);
            }
            ++ko;
        }
        if (qd == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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
    a.nQ64 = (L + BT - 1) / BT;
    a.scale = attn_scale;
    a.scale_log2 = attn_scale * kLog2e;
    a.status = status;
    float* lse2T = static_cast<float*>(ws);
    float* deltaT = lse2T + (size_t)B * H * a.Lp;
    a.lse2T = lse2T;
    a.deltaT = deltaT;
    const uint64_t cols = (uint64_t)H * 64;
    CUtensorMap q128, do128, k64, v64, dq128, k128, v128, q64, do64, dk128, dv128;
    if (!encode_bf16_seq(&q128, q, B, L, cols, BM) || !encode_bf16_seq(&do128, dout, B, L, cols, BM) ||
        !encode_bf16_seq(&k64, k, B, L, cols, BT) || !encode_bf16_seq(&v64, v, B, L, cols, BT) ||
        !encode_bf16_seq(&dq128, dq, B, L, cols, BM) || !encode_bf16_seq(&k128, k, B, L, cols, BM) ||
        !encode_bf16_seq(&v128, v, B, L, cols, BM) || !encode_bf16_seq(&q64, q, B, L, cols, BT) ||
        !encode_bf16_seq(&do64, dout, B, L, cols, BT) || !encode_bf16_seq(&dk128, dk, B, L, cols, BM) ||
        !encode_bf16_seq(&dv128, dv, B, L, cols, BM))
        return cudaErrorInvalidValue;
    const size_t nvec = (size_t)B * H * a.Lp;
    GCA_LAUNCH("swa_delta", st,
               swa_delta_kernel<<<(unsigned)((nvec + 255) / 256), 256, 0, st>>>(
                   static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse,
                   B, L, H, a.Lp, lse2T, deltaT));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

    a.n_items = B * a.nQT * H;
    int grid = a.n_items < sms ? a.n_items : sms;
    if ((e = cudaFuncSetAttribute(pa::swa_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  pa::SMEM)) != cudaSuccess)
        return e;
    GCA_LAUNCH("swa_bwd_q_tc", st,
               pa::swa_bwd_q_kernel<<<grid, kThreads, pa::SMEM, st>>>(q128, do128, k64, v64, dq128, a));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    a.n_items = B * a.nKT * H;
    grid = a.n_items < sms ? a.n_items : sms;
    if ((e = cudaFuncSetAttribute(pb::swa_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  pb::SMEM)) != cudaSuccess)
        return e;
    GCA_LAUNCH("swa_bwd_kv_tc", st,
               pb::swa_bwd_kv_kernel<<<grid, kThreads, pb::SMEM, st>>>(q64, do64, k128, v128, dk128,
                                                                       dv128, a));
    if ((e = cudaGetLastError()) == cudaSuccess) *launches += 3;
    return e;
}

}  // namespace gca
