// topk.cuh -- register top-k of a warp and 64-bit rank keys, shared by the
// scoring kernel and the decode retrieval.  Order everywhere: score
// descending, then index ascending (ties go to the lower chunk index).
#pragma once

#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace gca {

// Running top-k of a warp: lane j holds rank j (score desc, index asc); every
// lane also holds the current admission threshold (rank topk-1).
struct WarpTopk {
    float ts, thr_s;
    int ti, thr_i;
    __device__ void init() { ts = thr_s = -INFINITY; ti = thr_i = 0x7fffffff; }
    // (s, i) is uniform across the warp.
    __device__ __forceinline__ void offer(int topk, float s, int i) {
        if (!ranks_before(s, i, thr_s, thr_i)) return;
        const int lane = threadIdx.x & 31;
        const unsigned ahead = __ballot_sync(0xffffffffu, lane < topk && ranks_before(ts, ti, s, i));
        const int pos = __popc(ahead);
        const float us = __shfl_up_sync(0xffffffffu, ts, 1);
        const int ui = __shfl_up_sync(0xffffffffu, ti, 1);
        if (lane == pos) { ts = s; ti = i; }
        else if (lane > pos && lane < topk) { ts = us; ti = ui; }
        thr_s = __shfl_sync(0xffffffffu, ts, topk - 1);
        thr_i = __shfl_sync(0xffffffffu, ti, topk - 1);
    }
};

// Order-preserving key of a (score, index) pair: a larger key ranks earlier
// (higher score, then lower index; -0 and +0 are one score).  Keys of distinct
// indices are distinct, so
// the rank of a candidate in a set is the number of larger keys in it.  Key 0
// marks an empty list entry (it ranks after every real pair).
__device__ __forceinline__ unsigned long long rank_key(float f, int i) {
    unsigned u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;     // -0 ranks as +0 (they compare equal in ranks_before)
    const unsigned sk = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(sk) << 32) | static_cast<unsigned>(~static_cast<unsigned>(i));
}
__device__ __forceinline__ float key_score(unsigned long long k) {
    const unsigned sk = static_cast<unsigned>(k >> 32);
    return __uint_as_float((sk & 0x80000000u) ? (sk & 0x7fffffffu) : ~sk);
}
__device__ __forceinline__ int key_index(unsigned long long k) {
    return static_cast<int>(~static_cast<unsigned>(k & 0xffffffffull));
}

// Rank of key k among keys[0, n) (the number of larger keys), counted 32 keys
// per ballot by the whole warp (k uniform across it); stops at `limit`.
__device__ __forceinline__ int warp_rank(unsigned long long k, const unsigned long long* keys, int n,
                                         int limit) {
    const int lane = threadIdx.x & 31;
    int r = 0;
    for (int b0 = 0; b0 < n && r < limit; b0 += 32) {
        const int e = b0 + lane;
        r += __popc(__ballot_sync(0xffffffffu, e < n && keys[e] > k));
    }
    return r;
}

}  // namespace gca
