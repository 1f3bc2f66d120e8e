// MXFP8 quantisation (OCP Microscaling v1.0: E4M3 elements, one E8M0 scale
// per 32 consecutive elements along the contraction dimension).
//
// Layouts used by the library:
//   codes  : uint8 [rows, cols], row-major (cols = contraction dimension K)
//   scales : uint8 [groups, cols/32, ld_s] with rows split into `groups`
//            equal groups of rows_per_group (ld_s >= rows_per_group, a
//            multiple of 16 so that TMA can read whole scale columns);
//            byte = 127 + exponent of the block's power-of-two scale.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Quantise bf16 rows.  Source row of output row r: src_row_of ? src_row_of[r] /
// src_div : r (a gather, used to fuse the permutation).
cudaError_t launch_mx_quant_rows(const void* src, const int32_t* src_row_of, int src_div, int64_t rows, int cols,
                                 int64_t rows_per_group, int64_t ld_s, uint8_t* codes, uint8_t* scales,
                                 cudaStream_t st);

inline int64_t mx_scale_ld(int64_t rows) { return (rows + 15) / 16 * 16; }

}  // namespace moe
