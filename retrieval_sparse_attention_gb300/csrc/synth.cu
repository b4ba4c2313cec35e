// synth.cu -- device side of the counter-based synthetic input generator
// (SplitMix64 of Steele, Lea and Flood, OOPSLA 2014, used as a hash of the
// element counter).  Not part of GCA: it fills the large decode K/V cache
// directly in HBM so the host can regenerate any chunk of it for checking.
#include "common.cuh"
#include "gca_synth.h"
#include "kernels.h"

namespace gca {
namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <typename T>
__global__ void synth_fill_kernel(T* __restrict__ dst, size_t n, uint64_t key, uint64_t first) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t h = splitmix64(key ^ (first + i));
        const int s = (int)(h & 7) + (int)((h >> 3) & 7) + (int)((h >> 6) & 7) + (int)((h >> 9) & 7);
        dst[i] = from_f<T>((float)(s - 14) * (1.0f / 32.0f));
    }
}

}  // namespace

cudaError_t launch_synth_fill(void* dst, size_t n, gca_dtype_t dt, uint64_t seed, uint64_t tid,
                              uint64_t first, cudaStream_t st) {
    const uint64_t key = (seed << 56) ^ (tid << 48);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = sms > 0 ? sms * 8 : 1024;
    if (dt == GCA_BF16)
        GCA_LAUNCH("synth_fill", st, synth_fill_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>((__nv_bfloat16*)dst, n, key, first));
    else
        GCA_LAUNCH("synth_fill", st, synth_fill_kernel<float><<<blocks, 256, 0, st>>>((float*)dst, n, key, first));
    return cudaGetLastError();
}

}  // namespace gca
