// Host helper: TMA tensor maps for [outer][mid][inner] bf16 tensors.
#pragma once

#include <cuda.h>

namespace spc {

// Encodes a 3-D tiled map over a dense bf16 tensor of shape
// [outer][mid][inner] (inner contiguous) with 128-byte swizzle and zero fill
// outside the tensor.  box_inner * 2 bytes must be 128.  Returns an sp_status.
int encode_bf16_3d(CUtensorMap *map, const void *base, int inner, int mid, int outer, int box_inner, int box_mid,
                   int box_outer);

// Encodes a 2-D tiled map over a row-major bf16 matrix [rows][cols] (cols
// contiguous, cols * 2 a multiple of 16 bytes) with 128-byte swizzle and zero
// fill outside the matrix.  box_cols * 2 bytes must be 128; box_rows <= 256.
int encode_bf16_2d(CUtensorMap *map, const void *base, int cols, int rows, int box_cols, int box_rows);

}  // namespace spc
