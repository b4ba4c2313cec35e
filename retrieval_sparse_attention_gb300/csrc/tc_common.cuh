// tc_common.cuh -- helpers shared by the warp-specialised tensor-core kernels
// (forward, backward query-major pass, backward key-major pass).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace gca {
namespace tcx {

constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: far above any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Stage index + phase bit of a ring of mbarrier-guarded buffers.
struct Ring {
    int i;
    uint32_t ph;
    __device__ __forceinline__ void next(int n) {
        if (++i == n) { i = 0; ph ^= 1u; }
    }
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Two fp32 values as one 64-bit operand of the packed (f32x2) arithmetic, which
// issues one instruction for both lanes of the pair.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// bf16 pair from a packed pair (low half first)
__device__ __forceinline__ uint32_t pack_bf16x2(uint64_t v) {
    float lo, hi;
    f2_unpack(v, lo, hi);
    return pack_bf16(lo, hi);
}

__device__ __forceinline__ uint4 pack8(const float* x, float s) {
    return make_uint4(pack_bf16(x[0] * s, x[1] * s), pack_bf16(x[2] * s, x[3] * s),
                      pack_bf16(x[4] * s, x[5] * s), pack_bf16(x[6] * s, x[7] * s));
}

// pack8 with the scaling on column pairs (packed f32x2 multiply; the same roundings)
__device__ __forceinline__ uint4 pack8x2(const float* x, uint64_t s2) {
    return make_uint4(pack_bf16x2(fmul2(f2_pack(x[0], x[1]), s2)), pack_bf16x2(fmul2(f2_pack(x[2], x[3]), s2)),
                      pack_bf16x2(fmul2(f2_pack(x[4], x[5]), s2)), pack_bf16x2(fmul2(f2_pack(x[6], x[7]), s2)));
}

__device__ __forceinline__ uint4 pack8u(const uint32_t* r) {
    return make_uint4(pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1])),
                      pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3])),
                      pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5])),
                      pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7])));
}

// Bounded wait that also gives up once another role of the CTA has aborted:
// after `limit_ns` it records GCA_ERR_TIMEOUT, raises the CTA's abort flag and
// returns false.
__device__ __forceinline__ bool wait_bar_ns(int* abort_flag, uint64_t* bar, uint32_t parity,
                                            int* status, uint64_t limit_ns) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::global_timer_ns();
    while (true) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if (*((volatile int*)abort_flag)) return false;
        if (tc::global_timer_ns() - t0 > limit_ns) {
            set_status(status, GCA_ERR_TIMEOUT);
            *((volatile int*)abort_flag) = 1;
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar(int* abort_flag, uint64_t* bar, uint32_t parity,
                                         int* status) {
    return wait_bar_ns(abort_flag, bar, parity, status, kWaitNs);
}

// Address of the 16-byte chunk `ch` (0..7 within a 64-element row block) of
// row `row` in a K-major tile with the 128-byte swizzle (1024-byte aligned).
__device__ __forceinline__ uint32_t sw128_off(int row, int ch) {
    return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// MMA sequences with the operand descriptors built once: the start-address
// field holds (address >> 4) in the low 14 bits, so advancing an operand by
// B bytes adds B / 16 to the 64-bit descriptor (no carry: shared memory is
// below 256 KB).
// ---------------------------------------------------------------------------
// D (+)= A B^T over 64 elements of K (4 steps of 16), both operands K-major
// 128-byte-swizzled tiles whose rows are 128 bytes.
__device__ __forceinline__ void mma_kmajor_k64(uint32_t d, uint32_t a_addr, uint32_t b_addr,
                                               uint32_t idesc, uint32_t acc_first) {
    const uint64_t ad = tc::desc_kmajor_sw128(a_addr);
    const uint64_t bd = tc::desc_kmajor_sw128(b_addr);
    tc::mma_bf16(d, ad, bd, idesc, acc_first);
    tc::mma_bf16(d, ad + 2, bd + 2, idesc, 1);
    tc::mma_bf16(d, ad + 4, bd + 4, idesc, 1);
    tc::mma_bf16(d, ad + 6, bd + 6, idesc, 1);
}

// D (+)= P X over KSTEPS*16 elements of K: P K-major in blocks of 64 K
// elements (p_block bytes apart), X MN-major with 128-byte K rows.
template <int KSTEPS>
__device__ __forceinline__ void mma_kmajor_mnmajor(uint32_t d, uint32_t p_addr, uint32_t p_block,
                                                   uint32_t x_addr, uint32_t idesc,
                                                   uint32_t acc_first) {
    const uint64_t pd = tc::desc_kmajor_sw128(p_addr);
    const uint64_t xd = tc::desc_mnmajor_sw128(x_addr);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks)
        tc::mma_bf16(d, pd + (uint64_t)(((ks >> 2) * p_block + (ks & 3) * 32) >> 4),
                     xd + (uint64_t)(ks * 128), idesc, ks == 0 ? acc_first : 1u);
}

// ---------------------------------------------------------------------------
// Head tiles of DH = 32, 64 or 128 columns.  A [rows x DH] bf16 tile is held
// in shared memory as SUB sub-tiles, each [rows x SUB_COLS] with rows of
// ROW_BYTES bytes, exactly as one TMA box of SUB_COLS x rows writes it:
// DH = 64 and 128 use 64-column sub-tiles (128-byte rows, 128-byte swizzle),
// DH = 32 one 32-column tile (64-byte rows, 64-byte swizzle).  Sub-tile s of a
// tile whose sub-tiles hold R rows starts at s * R * ROW_BYTES.
// ---------------------------------------------------------------------------
template <int DH>
struct HeadGeom {
    static_assert(DH == 32 || DH == 64 || DH == 128, "head dimension 32, 64 or 128");
    static constexpr int SUB = DH == 128 ? 2 : 1;
    static constexpr int SUB_COLS = DH == 32 ? 32 : 64;
    static constexpr int ROW_BYTES = SUB_COLS * 2;
    static constexpr uint32_t SWZ = DH == 32 ? 4u : 2u;      // descriptor layout: 64B / 128B swizzle
    static constexpr uint32_t SBO = 8u * ROW_BYTES;           // bytes between 8-row groups
    static constexpr int KSTEPS_SUB = ROW_BYTES / 32;         // K = 16 steps along one row
    static constexpr uint32_t KROW16 = 16u * ROW_BYTES;       // bytes of 16 rows (MN-major K step)
    __host__ __device__ static constexpr int tile_bytes(int rows) { return rows * DH * 2; }
};

template <int DH>
__device__ __forceinline__ uint64_t desc_head(uint32_t saddr) {
    return tc::smem_desc(saddr, 16, HeadGeom<DH>::SBO, HeadGeom<DH>::SWZ);
}

// D (+)= A B^T contracted over the DH columns of two K-major head tiles whose
// sub-tiles hold a_rows and b_rows rows.
template <int DH>
__device__ __forceinline__ void mma_kmajor_dh(uint32_t d, uint32_t a_addr, int a_rows, uint32_t b_addr,
                                              int b_rows, uint32_t idesc, uint32_t acc_first) {
    using G = HeadGeom<DH>;
#pragma unroll
    for (int s = 0; s < G::SUB; ++s) {
        const uint64_t ad = desc_head<DH>(a_addr + s * a_rows * G::ROW_BYTES);
        const uint64_t bd = desc_head<DH>(b_addr + s * b_rows * G::ROW_BYTES);
#pragma unroll
        for (int ks = 0; ks < G::KSTEPS_SUB; ++ks)
            tc::mma_bf16(d, ad + 2 * ks, bd + 2 * ks, idesc, (s == 0 && ks == 0) ? acc_first : 1u);
    }
}

// D (+)= P X over KSTEPS*16 rows of K: P K-major (128-byte swizzle, blocks of 64
// K elements p_block bytes apart), X an MN-major head tile (K along its rows,
// x_rows rows per sub-tile).  Sub-tile s accumulates into TMEM columns
// d + s * SUB_COLS; idesc must give N = SUB_COLS.
template <int DH, int KSTEPS>
__device__ __forceinline__ void mma_kmajor_mn_dh(uint32_t d, uint32_t p_addr, uint32_t p_block,
                                                 uint32_t x_addr, int x_rows, uint32_t idesc,
                                                 uint32_t acc_first) {
    using G = HeadGeom<DH>;
    const uint64_t pd = tc::desc_kmajor_sw128(p_addr);
#pragma unroll
    for (int s = 0; s < G::SUB; ++s) {
        const uint64_t xd = desc_head<DH>(x_addr + s * x_rows * G::ROW_BYTES);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
            tc::mma_bf16(d + s * G::SUB_COLS, pd + (uint64_t)(((ks >> 2) * p_block + (ks & 3) * 32) >> 4),
                         xd + (uint64_t)(ks * (G::KROW16 >> 4)), idesc, ks == 0 ? acc_first : 1u);
    }
}

// D (+)= P X over KSTEPS*16 rows of K with P in tensor memory (p_tmem: column
// of K = 0, lane 0; 8 columns per K = 16 step) and X an MN-major head tile
// (x_rows rows per sub-tile).  Sub-tile s accumulates into TMEM columns
// d + s * SUB_COLS; idesc must give N = SUB_COLS and a K-major A.
template <int DH, int KSTEPS>
__device__ __forceinline__ void mma_ts_mn_dh(uint32_t d, uint32_t p_tmem, uint32_t x_addr, int x_rows,
                                             uint32_t idesc, uint32_t acc_first) {
    using G = HeadGeom<DH>;
#pragma unroll
    for (int s = 0; s < G::SUB; ++s) {
        const uint64_t xd = desc_head<DH>(x_addr + s * x_rows * G::ROW_BYTES);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
            tc::mma_bf16_ts(d + s * G::SUB_COLS, p_tmem + 8 * ks, xd + (uint64_t)(ks * (G::KROW16 >> 4)),
                            idesc, ks == 0 ? acc_first : 1u);
    }
}

// D (+)= A^T X over ksteps*16 rows of K: A MN-major with 128-byte rows (64
// elements along M), X an MN-major head tile (x_rows rows per sub-tile).
template <int DH>
__device__ __forceinline__ void mma_mn_mn_dh(uint32_t d, uint32_t a_addr, uint32_t x_addr, int x_rows,
                                             uint32_t idesc, int ksteps, uint32_t acc_first) {
    using G = HeadGeom<DH>;
    const uint64_t ad = tc::desc_mnmajor_sw128(a_addr);
#pragma unroll
    for (int s = 0; s < G::SUB; ++s) {
        const uint64_t xd = desc_head<DH>(x_addr + s * x_rows * G::ROW_BYTES);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            if (ks == ksteps) break;
            tc::mma_bf16(d + s * G::SUB_COLS, ad + (uint64_t)(ks * 128), xd + (uint64_t)(ks * (G::KROW16 >> 4)),
                         idesc, ks == 0 ? acc_first : 1u);
        }
    }
}

// Store DH fp32 TMEM columns of one accumulator row as bf16.  M = 64 layout
// (16x32bx2 reads): this thread holds half the row (u = 0: columns 0 .. DH/2-1,
// u = 1: the rest) of row lane%16 (+16 per lane quadrant); M = 128 layout: the
// whole row of its lane.
template <int M, int DH>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, __nv_bfloat16* dst_row, int u) {
    if constexpr (M == 64) {
        constexpr int HALF = DH / 2;
        uint32_t r[DH / 32][16];
#pragma unroll
        for (int i = 0; i < DH / 32; ++i) tc::tmem_ld_16x32bx2_x16<HALF>(taddr + 16 * i, r[i]);
        tc::tmem_wait_ld();
        uint4* dst = reinterpret_cast<uint4*>(dst_row + u * HALF);
#pragma unroll
        for (int i = 0; i < DH / 32; ++i) {
            dst[2 * i] = pack8u(r[i]);
            dst[2 * i + 1] = pack8u(r[i] + 8);
        }
    } else {
        uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
        for (int ci = 0; ci < DH / 16; ++ci) {
            uint32_t r[16];
            tc::tmem_ld_32x32b_x16(taddr + 16 * ci, r);
            tc::tmem_wait_ld();
            dst[2 * ci] = pack8u(r);
            dst[2 * ci + 1] = pack8u(r + 8);
        }
    }
}

// Zero one accumulator row's share (layout as store_acc_row).
template <int M, int DH>
__device__ __forceinline__ void zero_acc_row(__nv_bfloat16* dst_row, int u) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    constexpr int n16 = (M == 64 ? DH / 2 : DH) / 8;
    uint4* dst = reinterpret_cast<uint4*>(dst_row + (M == 64 ? u * (DH / 2) : 0));
#pragma unroll
    for (int q4 = 0; q4 < n16; ++q4) dst[q4] = z;
}

// Untiled bulk copy global -> shared, completing on an mbarrier (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

}  // namespace tcx
}  // namespace gca
