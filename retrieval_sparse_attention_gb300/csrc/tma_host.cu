// tma_host.cu -- encoding of TMA tensor maps (cuTensorMapEncodeTiled, taken
// from the driver through the runtime's entry-point query, so the library
// does not link libcuda directly).
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "tma_host.h"

namespace gca {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_once;

void resolve() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}

}  // namespace

bool encode_bf16_rows_box(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                          uint32_t box_cols, uint32_t box_rows) {
    std::call_once(g_once, resolve);
    if (!g_encode || (box_cols != 64 && box_cols != 32)) return false;
    // 2-D view [rows, row_elems] of bf16, box = box_cols x box_rows, written to
    // shared memory with the swizzle whose span is one box row (128 or 64 bytes).
    cuuint64_t dims[2] = {row_elems, rows};
    cuuint64_t strides[1] = {row_elems * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                      uint32_t box_rows) {
    return encode_bf16_rows_box(map, base, rows, row_elems, 64, box_rows);
}

bool encode_bf16_seq(CUtensorMap* map, const void* base, uint64_t B, uint64_t L, uint64_t row_elems,
                     uint32_t box_rows) {
    std::call_once(g_once, resolve);
    if (!g_encode) return false;
    cuuint64_t dims[3] = {row_elems, L, B};
    cuuint64_t strides[2] = {row_elems * 2, L * row_elems * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_f32_box(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                    uint32_t box_cols, uint32_t box_rows) {
    std::call_once(g_once, resolve);
    if (!g_encode) return false;
    cuuint64_t dims[2] = {row_elems, rows};
    cuuint64_t strides[1] = {row_elems * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gca
