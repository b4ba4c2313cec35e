// tma_host.h -- host-side TMA tensor-map encoding used by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gca {

// Tensor map over a row-major bf16 matrix [rows, row_elems] (row stride
// row_elems * 2 bytes, a multiple of 16), box of 64 columns x box_rows rows,
// 128-byte swizzle.  Returns false if the driver entry point is missing or
// rejects the arguments.
bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                      uint32_t box_rows);

// The same view with a box of box_cols (64 or 32) columns: 64 columns use the
// 128-byte swizzle, 32 columns the 64-byte swizzle (one box row per swizzle span).
bool encode_bf16_rows_box(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                          uint32_t box_cols, uint32_t box_rows);

// Tensor map over bf16 sequences [B, L, row_elems] (row stride row_elems * 2
// bytes, a multiple of 16), box of 64 columns x box_rows rows x 1 sequence,
// 128-byte swizzle.  Rows outside [0, L) of a sequence are out of bounds:
// loads fill them with zeros, stores skip them.
bool encode_bf16_seq(CUtensorMap* map, const void* base, uint64_t B, uint64_t L, uint64_t row_elems,
                     uint32_t box_rows);

// Tensor map over a row-major fp32 matrix [rows, row_elems] (row stride
// row_elems * 4 bytes, a multiple of 16), box of box_cols x box_rows (box_cols
// * 4 a multiple of 16), no swizzle: the box lands in shared memory as
// box_rows dense rows of box_cols floats.
bool encode_f32_box(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                    uint32_t box_cols, uint32_t box_rows);

}  // namespace gca
