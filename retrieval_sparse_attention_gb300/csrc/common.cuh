// common.cuh -- shared device helpers of the GCA CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gca.h"

namespace gca {

// ---------------------------------------------------------------------------
// Element conversion
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// Device status word: set once by the first error, read by gca_get_status().
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Ranking used by every top-k: larger score first, then smaller index.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool ranks_before(float s1, int i1, float s2, int i2) {
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Upper bound on top-k handled by the kernels (one warp lane per rank).
constexpr int kMaxTopk = 32;

// Host-side launch bookkeeping (per host thread).
void note_launches(int n);
void reset_launches();

}  // namespace gca
