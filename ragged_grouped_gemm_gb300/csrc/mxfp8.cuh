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

// Quantise bf16 matrices along their ROWS (the contraction runs over rows)
// and write the codes transposed, so that the contraction becomes the
// contiguous (K-major) axis of the output:
//   src    : `batch` matrices [rows, cols] (batch stride rows*cols); row r of
//            a matrix is source row src_row_of[r] / src_div when src_row_of
//            is given (a gather, used to read x in permuted order)
//   codes  : [batch][cols][ld_codes]  (block j of 32 rows -> bytes 32j..32j+31)
//   scales : [batch][ld_codes/32][ld_s]
// Without `offsets` the blocks are consecutive 32-row blocks of each matrix
// (ld_codes >= rows).  With `offsets` (batch 1, n_groups ragged row groups of
// the expert-major buffer) the blocks restart at every group's first row and
// group g occupies output positions pad_offsets[g] .. pad_offsets[g+1]-1,
// its row count rounded up to a multiple of 128 with zero codes.
cudaError_t launch_mx_quant_cols_t(const void* src, int64_t batch, int64_t rows, int cols,
                                   const int32_t* src_row_of, int src_div, const int32_t* offsets,
                                   const int32_t* pad_offsets, int n_groups, int64_t ld_codes, uint8_t* codes,
                                   int64_t ld_s, uint8_t* scales, cudaStream_t st);

// FP8 weights with per-tile scaling: codes [batch][rows][cols] E4M3 and
// scales [batch][ceil(rows/128)][ceil(cols/128)] fp32, scale = amax / 448 of
// the 128 x 128 tile (1 for an all-zero tile), code = E4M3(w / scale), the
// quotient formed in double and rounded once (nearest even, saturating).
cudaError_t launch_fp8_tile_quant(const void* src, int64_t batch, int64_t rows, int64_t cols, uint8_t* codes,
                                  float* scales, cudaStream_t st);

// pad_offsets[g] = sum over g' < g of ceil(count_g' / 128) * 128 (n_groups + 1 entries).
cudaError_t launch_pad_offsets(const int32_t* offsets, int n_groups, int32_t* pad_offsets, cudaStream_t st);

// Upper bound of pad_offsets[n_groups] for `rows` rows in `n_groups` groups.
inline int64_t mx_padded_rows(int64_t rows, int n_groups) { return (rows + 127) / 128 * 128 + 128LL * n_groups; }

}  // namespace moe
