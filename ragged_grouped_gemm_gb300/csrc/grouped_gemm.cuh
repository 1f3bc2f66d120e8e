// Host-side interface of the persistent tcgen05 grouped GEMM.
//
// One launch computes, for every group g of a ragged problem,
//   C_g = A_g * B_g^T       (A_g: [m_g, K], B_g: [N, K], fp32 accumulation)
// where the ragged dimension is either M (forward and data-gradient GEMMs:
// the rows of expert g in the expert-major permuted buffers) or K (weight
// gradients: the contraction runs over the rows of expert g).  Group sizes
// are read on the device from an offsets array, so no host synchronisation
// and no padding is needed ("Accelerating Dropless MoE Training in JAX with
// NVIDIA Transformer Engine", ¶5-¶6: grouped GEMM over ragged tensors in a
// single call, with shapes not known on the CPU).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

enum EpiKind : int {
  EPI_BF16 = 0,        // out0[row, col] = bf16(acc)
  EPI_F32 = 1,         // out0[row, col] = acc
  EPI_SWIGLU_FWD = 2,  // acc = [a1 | a3] -> out0 = h = silu(a1) * a3, out1 = a1, out2 = a3 (bf16)
  EPI_SWIGLU_BWD = 3,  // acc = dh; in0 = a1, in1 = a3 -> out0 = da1, out1 = da3 (bf16)
  EPI_SWIGLU_FWD_Q = 4,  // acc = [a1 | a3] -> h quantised to MXFP8 along F: out0 = codes [rows, n],
                         // out1 = scales [n/32, s_ld]; optional bf16 out2 = h, out3 = a1, out4 = a3
};

// MXFP8 operand: E4M3 codes [groups][rows, cols] and E8M0 scales
// [groups][cols/32, scale_ld] (see mxfp8.cuh), cols = contraction dimension.
struct MxOperand {
  const void* codes = nullptr;
  const void* scales = nullptr;
  int64_t rows = 0;
  int64_t cols = 0;
  int64_t groups = 1;
  int64_t scale_ld = 0;
};

// One operand source: a bf16 matrix in global memory.
//   K-major A: [rows, K] row-major (rows = permuted rows), ld = K.
//   K-major B: per group [N, K] row-major, groups stacked with group_stride.
//   MN-major A/B: [K_rows, MN] row-major (the contraction runs over rows).
struct Operand {
  const void* ptr = nullptr;
  int64_t rows = 0;          // per group for stacked weights
  int64_t cols = 0;
  int64_t ld = 0;            // elements between consecutive rows
  int64_t groups = 1;        // >1: a stack of matrices (3-D tensor map)
  int64_t group_stride = 0;  // elements between consecutive matrices
};

struct GemmArgs {
  bool a_mn = false;          // A stored MN-major (weight gradients)
  bool b_mn = false;          // B stored MN-major (data gradients)
  bool ragged_k = false;      // contraction over the group's rows
  int block_n = 256;          // 256, or 32 for narrow N (router logits)
  int ksplit = 1;             // one group, fp32 out: the contraction in ksplit slices, out0 =
                              // [ksplit][rows][ld_out] partial products (summed by the caller)
  EpiKind epi = EPI_BF16;
  Operand a[2];               // a[1]: second half of a split contraction
  Operand b[2];               // b[1]: second contraction half, or W3 half of the N tile
  bool b_dual_n = false;      // N tile = [b[0] rows | b[1] rows] (fused W1|W3)
  int k0 = 0, k1 = 0;         // ragged M: contraction length of source 0 and 1
  const int32_t* offsets = nullptr;  // device, [num_groups + 1]
  int num_groups = 1;
  int64_t max_rows = 0;       // upper bound of offsets[num_groups] (grid sizing)
  int m_size = 0;             // ragged K: rows of each C_g
  int n_size = 0;             // columns of C (f extent for EPI_SWIGLU_FWD)
  bool quant = false;         // operands are MXFP8 (qa, qb), dequantised to bf16 on the way in
  MxOperand qa[2];            // A per contraction source: [rows, K] with scales [K/32, scale_ld]
                              // (ragged K: [M, K_padded] with scales [K_padded/32, scale_ld])
  MxOperand qb[2];            // B: [groups][N, K]; qb[1] is the W3 half of a dual-N tile
  void* out0 = nullptr;
  void* out1 = nullptr;
  void* out2 = nullptr;
  void* out3 = nullptr;
  void* out4 = nullptr;
  int64_t s_ld = 0;           // EPI_SWIGLU_FWD_Q: leading dimension of the h scales
  const void* in0 = nullptr;
  const void* in1 = nullptr;
  int64_t ld_out = 0;
  int64_t group_stride_out = 0;
  int32_t* status = nullptr;  // device status words
  // FP8 weights (bf16 A): b[] hold E4M3 codes (uint8, ld and group_stride in
  // bytes) of weight matrices [rows][cols] (K-major B: rows = n; MN-major B:
  // rows = k) and w8_scale[] their fp32 scales per 128 x 128 tile,
  // [groups][ceil(rows/128)][ceil(cols/128)]; dequantised to bf16 in shared memory
  bool w8 = false;
  const float* w8_scale[2] = {nullptr, nullptr};
  // Gathered A (ragged M, K-major bf16, one contraction source): row r of the
  // problem is row a_gather[r] / gather_k of a[0] (the token matrix [N, K0]),
  // loaded by TMA tile::gather4 instead of a permuted copy
  const int32_t* a_gather = nullptr;
  int gather_k = 0;
  // Ragged K (bf16) with several groups: global scratch of
  // kGemmMapScratchBytes, 128-byte aligned, for the per-group tensor maps a
  // small kernel writes before the GEMM (same stream)
  void* map_ws = nullptr;
};

// Scratch the ragged-K bf16 form needs in GemmArgs::map_ws: two 128-byte
// tensor maps per group (at most 1024 groups).
constexpr size_t kGemmMapScratchBytes = 2 * 1024 * 128;

// Enqueue the grouped GEMM on `stream`.  Returns cudaSuccess or the first
// CUDA error (tensor-map encoding failures map to cudaErrorInvalidValue).
cudaError_t launch_grouped_gemm(const GemmArgs& args, cudaStream_t stream);

int num_sms();
// Contraction slices a launch with GemmArgs::ksplit = requested over k
// elements actually uses (slices of whole 64-element k-blocks, none empty).
int gemm_ksplit(int64_t k, int requested);

}  // namespace moe
