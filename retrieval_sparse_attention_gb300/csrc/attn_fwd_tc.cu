// attn_fwd_tc.cu -- GCA forward on the Blackwell tensor cores (bf16, d = 64).
//
// GCA (README "Model Architecture"; Figure 1/2; Eq. 2 as the batch form of
// Figure 2): every token t of query chunk c attends separately to each
// retrieved chunk kappa_j (stage 1), O_t^j = softmax(s q_t K_j^T) V_j, and the
// outputs are fused as O_t = sum_j w_j O_t^j (stage 2).  App. B: the forward
// also returns the log-sum-exp of every (token, slot).
//
// Design (one persistent CTA per SM, 6 warps, warp-specialised):
//   warp 0     TMA producer: Q tile of the work item, then the K and V tiles of
//              each retrieved chunk, gathered straight from the [tokens, H*d]
//              tensors (box 64 x S, 128-byte swizzle) into a ring of stages.
//   warp 1     MMA issuer (one thread) and TMEM owner: S_g = Q K_g^T for a
//              group of retrieved chunks (N = 128 keys), then O += P_g V_g.
//   warps 2-5  softmax + epilogue: read S_g from TMEM, per-slot max / sum /
//              exp2, write P_g = exp(S - m) * (w_j / l_j) as bf16 into shared
//              memory (the A operand of the PV MMA), write the lse; at the end
//              of the item read O from TMEM and store it as bf16.
// Because each slot's softmax is normalised before PV and carries its fusion
// weight, the per-slot outputs O_t^j are summed by the tensor core in TMEM
// and never exist in memory.  A work item is (batch row, query chunk, head).
//
// S = 64 : M = 64 MMAs (TMEM rows r at lanes r%16 + 32*(r/16)); a group is two
//          slots; each softmax thread owns one (token, slot) row of 64 keys.
// S = 128: M = 128 MMAs (row r at lane r); a group is one slot; each softmax
//          thread owns one token row of 128 keys.
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

constexpr int kThreads = 192;
using tcx::Ring;
using tcx::fast_exp2;
using tcx::pack_bf16;
using tcx::kLog2e;
using tcx::kLn2;

template <int S>
struct Cfg {
    static constexpr int M = S;                         // tokens per item = MMA M
    static constexpr int GS = 128 / S;                  // slots per group
    static constexpr int NG = 128;                      // keys per full group
    static constexpr int STAGES = (S == 64) ? 4 : 3;    // K/V ring depth
    static constexpr int TILE = S * 128;                // one slot's K (or V) tile, bytes
    static constexpr int Q_BYTES = S * 128;
    static constexpr int STAGE_BYTES = 2 * NG * 128;    // K half then V half
    static constexpr int P_BLOCK = M * 128;             // 64 keys of P for all M rows
    static constexpr int P_BYTES = M * NG * 2;
    static constexpr int VALS = (S == 64) ? 64 : 128;   // S values per softmax thread
    // shared-memory carve-up (all 1024-byte aligned)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_P = OFF_KV + STAGES * STAGE_BYTES;
    static constexpr int SMEM = OFF_P + 2 * P_BYTES + 1024;   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;                // two S buffers of 128 columns
    static constexpr uint32_t COL_O = 256;              // two O buffers of 64 columns
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

struct __align__(8) Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[4], kv_empty[4];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t done;
    uint32_t tmem;
    int abort;
};

// Valid slots of one item: slot numbers and their chunks, in slot order.
__device__ __forceinline__ int item_slots(const FwdArgs& a, int b, int c, int* js, int* kaps,
                                          bool report) {
    const int32_t* row = a.idx + ((size_t)b * a.nQ + c) * a.topk;
    int n = 0;
    for (int j = 0; j < a.topk; ++j) {
        const int kap = row[j];
        if (kap >= 0 && kap < a.nP) { js[n] = j; kaps[n] = kap; ++n; }
        else if (kap >= a.nP && report) set_status(a.status, GCA_ERR_DEVICE_INDEX);
    }
    return n;
}

__device__ __forceinline__ bool wait_bar(Bars& sb, uint64_t* bar, uint32_t parity, int* status) {
    return tcx::wait_bar(&sb.abort, bar, parity, status);
}

template <int S>
__global__ void __launch_bounds__(kThreads, 1)
gca_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
    using C = Cfg<S>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ Bars sb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&sb.kv_full[i], 1);
            mbar_init(&sb.kv_empty[i], 1);
        }
        mbar_init(&sb.done, 1);
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
    int js[kMaxTopk], kaps[kMaxTopk];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            Ring kv{0, 0}, qr{0, 0};
            bool kv_out[4] = {false, false, false, false}, q_out[2] = {false, false};
            uint32_t kv_ph[4] = {0, 0, 0, 0}, q_ph[2] = {0, 0};
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                const int h = item % a.H, bc = item / a.H, c = bc % a.nQ, b = bc / a.nQ;
                const int n = item_slots(a, b, c, js, kaps, true);
                if (n == 0) continue;
                if (!wait_bar(sb, &sb.q_empty[qr.i], qr.ph ^ 1u, a.status)) break;
                mbar_arrive_expect_tx(&sb.q_full[qr.i], C::Q_BYTES);
                tma_load_2d(sm + C::OFF_Q + qr.i * C::Q_BYTES, &tq, &sb.q_full[qr.i], h * 64,
                            b * a.Lq + c * S);
                q_out[qr.i] = true;
                q_ph[qr.i] = qr.ph;
                qr.next(2);
                bool ok = true;
                for (int g = 0; g * C::GS < n; ++g) {
                    const int ns = min(C::GS, n - g * C::GS);
                    if (!wait_bar(sb, &sb.kv_empty[kv.i], kv.ph ^ 1u, a.status)) { ok = false; break; }
                    uint8_t* stg = sm + C::OFF_KV + kv.i * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&sb.kv_full[kv.i], ns * 2 * C::TILE);
                    for (int u = 0; u < ns; ++u) {
                        const int y = (b * a.nP + kaps[g * C::GS + u]) * S;
                        tma_load_2d(stg + u * C::TILE, &tk, &sb.kv_full[kv.i], h * 64, y);
                        tma_load_2d(stg + C::NG * 128 + u * C::TILE, &tv, &sb.kv_full[kv.i],
                                    h * 64, y);
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
            for (int i = 0; i < 2; ++i)
                if (q_out[i]) mbar_wait(&sb.q_full[i], q_ph[i], nullptr, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            Ring kv{0, 0}, qr{0, 0}, s{0, 0}, p{0, 0}, o{0, 0};
            bool issued = false;
            const uint32_t id_s128 = idesc_bf16(C::M, 128, false, false);
            const uint32_t id_s64 = idesc_bf16(C::M, 64, false, false);
            const uint32_t id_o = idesc_bf16(C::M, 64, false, true);
            for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
                const int h = item % a.H, bc = item / a.H, c = bc % a.nQ, b = bc / a.nQ;
                (void)h;
                const int n = item_slots(a, b, c, js, kaps, false);
                if (n == 0) continue;
                const int G = (n + C::GS - 1) / C::GS;
                if (!wait_bar(sb, &sb.q_full[qr.i], qr.ph, a.status)) break;
                if (!wait_bar(sb, &sb.o_empty[o.i], o.ph ^ 1u, a.status)) break;
                tc_fence_after();
                const uint32_t qaddr = smem_u32(sm + C::OFF_Q + qr.i * C::Q_BYTES);
                const uint32_t d_o = tmem + C::COL_O + o.i * 64;
                int stg_of[2] = {0, 0};
                auto issue_s = [&](int g) -> bool {
                    const int ns = min(C::GS, n - g * C::GS);
                    if (!wait_bar(sb, &sb.kv_full[kv.i], kv.ph, a.status)) return false;
                    if (!wait_bar(sb, &sb.s_empty[s.i], s.ph ^ 1u, a.status)) return false;
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(sm + C::OFF_KV + kv.i * C::STAGE_BYTES);
                    const uint32_t d = tmem + C::COL_S + s.i * 128;
                    const uint32_t id = (ns * S == 128) ? id_s128 : id_s64;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(d, desc_kmajor_sw128(qaddr + 32 * ks),
                                 desc_kmajor_sw128(kaddr + 32 * ks), id, ks > 0);
                    mma_commit(&sb.s_full[s.i]);
                    stg_of[g & 1] = kv.i;
                    kv.next(C::STAGES);
                    s.next(2);
                    issued = true;
                    return true;
                };
                bool ok = issue_s(0);
                for (int g = 0; ok && g < G; ++g) {
                    if (g + 1 < G && !issue_s(g + 1)) { ok = false; break; }
                    const int ns = min(C::GS, n - g * C::GS);
                    if (!wait_bar(sb, &sb.p_full[p.i], p.ph, a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t paddr = smem_u32(sm + C::OFF_P + p.i * C::P_BYTES);
                    const uint32_t vaddr =
                        smem_u32(sm + C::OFF_KV + stg_of[g & 1] * C::STAGE_BYTES + C::NG * 128);
                    const int ksteps = ns * S / 16;
                    for (int ks = 0; ks < ksteps; ++ks)
                        mma_bf16(d_o, desc_kmajor_sw128(paddr + (ks >> 2) * C::P_BLOCK + (ks & 3) * 32),
                                 desc_mnmajor_sw128(vaddr + ks * 2048), id_o, (g > 0 || ks > 0));
                    mma_commit(&sb.kv_empty[stg_of[g & 1]]);
                    mma_commit(&sb.p_empty[p.i]);
                    p.next(2);
                }
                if (!ok) break;
                mma_commit(&sb.o_full[o.i]);
                mma_commit(&sb.q_empty[qr.i]);
                o.next(2);
                qr.next(2);
            }
            if (issued) {
                // every MMA must have finished before TMEM is released
                mma_commit(&sb.done);
                mbar_wait(&sb.done, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int qd = warp & 3;
        const int row = (S == 64) ? 16 * qd + (lane & 15) : 32 * qd + lane;
        const int u = (S == 64) ? (lane >> 4) : 0;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        Ring s{0, 0}, p{0, 0}, o{0, 0};
        for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
            const int h = item % a.H, bc = item / a.H, c = bc % a.nQ, b = bc / a.nQ;
            const int n = item_slots(a, b, c, js, kaps, false);
            const size_t tok = (size_t)b * a.Lq + (size_t)c * S + row;
            const int32_t* irow = a.idx + ((size_t)b * a.nQ + c) * a.topk;
            const float* wrow = a.w + ((size_t)b * a.nQ + c) * a.topk;
            __nv_bfloat16* orow = a.o + (tok * a.H + h) * 64;
            float* lrow = a.lse ? a.lse + (tok * a.H + h) * a.topk : nullptr;
            if (lrow && u == 0)
                for (int j = 0; j < a.topk; ++j) {
                    const int kap = irow[j];
                    if (kap < 0) lrow[j] = -INFINITY;
                    else if (kap >= a.nP) lrow[j] = NAN;
                }
            if (n == 0) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                if (S == 64) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) reinterpret_cast<uint4*>(orow + u * 32)[q4] = z;
                } else {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) reinterpret_cast<uint4*>(orow)[q4] = z;
                }
                continue;
            }
            bool ok = true;
            for (int g = 0; g * C::GS < n; ++g) {
                const int ns = min(C::GS, n - g * C::GS);
                const bool active = u < ns;
                if (!wait_bar(sb, &sb.s_full[s.i], s.ph, a.status)) { ok = false; break; }
                tc_fence_after();
                float x[C::VALS];
                const uint32_t taddr = tmem + lane_base + C::COL_S + s.i * 128;
                if (S == 64) {
#pragma unroll
                    for (int ci = 0; ci < C::VALS / 16; ++ci) {
                        uint32_t r[16];
                        tmem_ld_16x32bx2_x16<64>(taddr + 16 * ci, r);
#pragma unroll
                        for (int t = 0; t < 16; ++t) x[16 * ci + t] = __uint_as_float(r[t]);
                    }
                } else {
#pragma unroll
                    for (int ci = 0; ci < C::VALS / 16; ++ci) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(taddr + 16 * ci, r);
#pragma unroll
                        for (int t = 0; t < 16; ++t) x[16 * ci + t] = __uint_as_float(r[t]);
                    }
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sb.s_empty[s.i]);
                s.next(2);
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < C::VALS; ++i) mx = fmaxf(mx, x[i]);
                const float mb = mx * a.scale_log2;
                float l = 0.f;
#pragma unroll
                for (int i = 0; i < C::VALS; ++i) {
                    x[i] = fast_exp2(fmaf(x[i], a.scale_log2, -mb));
                    l += x[i];
                }
                float coef = 0.f;
                if (active) {
                    const int j = js[g * C::GS + u];
                    coef = wrow[j] / l;
                    if (lrow) lrow[j] = (mb + log2f(l)) * kLn2;
                }
                if (!wait_bar(sb, &sb.p_empty[p.i], p.ph ^ 1u, a.status)) { ok = false; break; }
                if (active) {
                    uint8_t* pbase = sm + C::OFF_P + p.i * C::P_BYTES + row * 128;
#pragma unroll
                    for (int ch = 0; ch < C::VALS / 8; ++ch) {
                        uint4 v;
                        v.x = pack_bf16(x[8 * ch + 0] * coef, x[8 * ch + 1] * coef);
                        v.y = pack_bf16(x[8 * ch + 2] * coef, x[8 * ch + 3] * coef);
                        v.z = pack_bf16(x[8 * ch + 4] * coef, x[8 * ch + 5] * coef);
                        v.w = pack_bf16(x[8 * ch + 6] * coef, x[8 * ch + 7] * coef);
                        const int blk = (S == 64) ? u : (ch >> 3);
                        const int cc = ch & 7;
                        *reinterpret_cast<uint4*>(pbase + blk * C::P_BLOCK + ((cc ^ (row & 7)) << 4)) = v;
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&sb.p_full[p.i]);
                p.next(2);
            }
            if (!ok) break;
            if (!wait_bar(sb, &sb.o_full[o.i], o.ph, a.status)) break;
            tc_fence_after();
            const uint32_t oaddr = tmem + lane_base + C::COL_O + o.i * 64;
            if (S == 64) {
                uint32_t r0[16], r1[16];
                tmem_ld_16x32bx2_x16<32>(oaddr, r0);
                tmem_ld_16x32bx2_x16<32>(oaddr + 16, r1);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sb.o_empty[o.i]);
                uint4* dst = reinterpret_cast<uint4*>(orow + u * 32);
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    dst[q4] = make_uint4(pack_bf16(__uint_as_float(r0[8 * q4 + 0]), __uint_as_float(r0[8 * q4 + 1])),
                                         pack_bf16(__uint_as_float(r0[8 * q4 + 2]), __uint_as_float(r0[8 * q4 + 3])),
                                         pack_bf16(__uint_as_float(r0[8 * q4 + 4]), __uint_as_float(r0[8 * q4 + 5])),
                                         pack_bf16(__uint_as_float(r0[8 * q4 + 6]), __uint_as_float(r0[8 * q4 + 7])));
                    dst[2 + q4] = make_uint4(pack_bf16(__uint_as_float(r1[8 * q4 + 0]), __uint_as_float(r1[8 * q4 + 1])),
                                             pack_bf16(__uint_as_float(r1[8 * q4 + 2]), __uint_as_float(r1[8 * q4 + 3])),
                                             pack_bf16(__uint_as_float(r1[8 * q4 + 4]), __uint_as_float(r1[8 * q4 + 5])),
                                             pack_bf16(__uint_as_float(r1[8 * q4 + 6]), __uint_as_float(r1[8 * q4 + 7])));
                }
            } else {
                uint32_t r[4][16];
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) tmem_ld_32x32b_x16(oaddr + 16 * ci, r[ci]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&sb.o_empty[o.i]);
                uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
                for (int ci = 0; ci < 4; ++ci)
#pragma unroll
                    for (int q4 = 0; q4 < 2; ++q4)
                        dst[2 * ci + q4] = make_uint4(
                            pack_bf16(__uint_as_float(r[ci][8 * q4 + 0]), __uint_as_float(r[ci][8 * q4 + 1])),
                            pack_bf16(__uint_as_float(r[ci][8 * q4 + 2]), __uint_as_float(r[ci][8 * q4 + 3])),
                            pack_bf16(__uint_as_float(r[ci][8 * q4 + 4]), __uint_as_float(r[ci][8 * q4 + 5])),
                            pack_bf16(__uint_as_float(r[ci][8 * q4 + 6]), __uint_as_float(r[ci][8 * q4 + 7])));
            }
            o.next(2);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg<S>::TMEM_COLS);
    }
}

template <int S>
cudaError_t launch_s(const Shape& sp, const void* q, const void* k, const void* v,
                     const int32_t* idx, const float* w, void* o, float* lse, int* status,
                     cudaStream_t st) {
    CUtensorMap tq, tk, tv;
    const uint64_t cols = (uint64_t)sp.H * 64;
    if (!encode_bf16_rows(&tq, q, (uint64_t)sp.B * sp.Lq, cols, S) ||
        !encode_bf16_rows(&tk, k, (uint64_t)sp.B * sp.nP * S, cols, S) ||
        !encode_bf16_rows(&tv, v, (uint64_t)sp.B * sp.nP * S, cols, S))
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
    auto kern = gca_fwd_tc_kernel<S>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<S>::SMEM);
    if (e != cudaSuccess) return e;
    GCA_LAUNCH("fwd_tc", st, kern<<<grid, kThreads, Cfg<S>::SMEM, st>>>(tq, tk, tv, a));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const Shape& sp, const void* q, const void* k, const void* v,
                          const int32_t* idx, const float* w, void* o, float* lse, int* status,
                          cudaStream_t st, int* launches) {
    cudaError_t e = (sp.S == 64) ? launch_s<64>(sp, q, k, v, idx, w, o, lse, status, st)
                                 : launch_s<128>(sp, q, k, v, idx, w, o, lse, status, st);
    if (e == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace gca
