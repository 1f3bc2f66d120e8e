// MXFP8 quantisation kernels.  Row-wise: one thread per (row, 32-element
// block), a warp covering 32 consecutive blocks of one row, so the warp
// reads 2 KB and writes 1 KB of codes contiguously.
//
// Scale rule (OCP MX v1.0 with E4M3 elements, emax = 8): the block's shared
// scale is 2^(floor(log2(amax)) - 8), clamped to [2^-127, 2^127]; an all-zero
// block gets 2^-127 and zero codes.  floor(log2(amax)) is read from amax's
// exponent bits (leading-bit position for a subnormal amax).  Elements are
// divided by the scale (an exact power-of-two multiply) and converted to E4M3
// with round-to-nearest-even and saturation at +-448 (cvt.rn.satfinite).
#include "mxfp8.cuh"

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "mx_device.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) mx_quant_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                            const int32_t* __restrict__ src_row_of, int src_div,
                                                            int64_t rows, int cols, int64_t rows_per_group,
                                                            int64_t ld_s, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales) {
  const int nkb = cols / 32;
  const int chunks = (nkb + 31) / 32;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t row = w / chunks;
  const int kb = static_cast<int>(w - row * chunks) * 32 + (threadIdx.x & 31);
  if (row >= rows || kb >= nkb) return;
  const int64_t sr = src_row_of ? src_row_of[row] / src_div : row;
  const uint4* p = reinterpret_cast<const uint4*>(src + sr * cols + kb * 32);
  const uint4 v[4] = {p[0], p[1], p[2], p[3]};
  uint4 c0, c1;
  const uint8_t sc = mx_quant_block32(v, c0, c1);
  uint4* dst = reinterpret_cast<uint4*>(codes + row * cols + kb * 32);
  dst[0] = c0;
  dst[1] = c1;
  const int64_t g = row / rows_per_group;
  const int64_t n = row - g * rows_per_group;
  scales[(g * nkb + kb) * ld_s + n] = sc;
}

// Transposing quantiser.  One CTA: one output block of 32 quantised rows x
// 128 columns.  The 32 x 128 bf16 tile is staged in shared memory with
// coalesced 16-byte loads (16 threads per 256-byte row segment); thread t
// then quantises column t and writes its 32 codes with one 32-byte store.
__global__ void __launch_bounds__(128) mx_quant_cols_t_kernel(
    const __nv_bfloat16* __restrict__ src, int64_t rows, int cols, const int32_t* __restrict__ src_row_of,
    int src_div, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pad_offsets, int n_groups,
    int64_t ld_codes, uint8_t* __restrict__ codes, int64_t ld_s, uint8_t* __restrict__ scales) {
  __shared__ __align__(16) __nv_bfloat16 tile[32][128 + 8];   // +8: rows 16 B apart in the bank pattern
  const int64_t jb = blockIdx.x;
  const int b = blockIdx.z;
  const int c0 = blockIdx.y * 128;
  int64_t r0, nvalid;
  if (offsets) {
    const int64_t p0 = jb * 32;
    if (p0 >= pad_offsets[n_groups]) return;   // uniform across the block
    int lo = 0, hi = n_groups;   // largest g with pad_offsets[g] <= p0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pad_offsets[mid] <= p0) lo = mid; else hi = mid;
    }
    r0 = offsets[lo] + (p0 - pad_offsets[lo]);
    nvalid = max(int64_t{0}, min(int64_t{32}, static_cast<int64_t>(offsets[lo + 1]) - r0));
  } else {
    r0 = jb * 32;
    nvalid = max(int64_t{0}, min(int64_t{32}, rows - r0));
  }
  const __nv_bfloat16* m = src + static_cast<int64_t>(b) * rows * cols;
  // stage: 32 rows x 16 chunks of 8 bf16; cols is a multiple of 8
  for (int i = threadIdx.x; i < 32 * 16; i += 128) {
    const int rr = i >> 4, ch = i & 15;
    const int c = c0 + ch * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (rr < nvalid && c < cols) {
      const int64_t r = r0 + rr;
      const int64_t sr = src_row_of ? src_row_of[r] / src_div : r;
      v = *reinterpret_cast<const uint4*>(m + sr * cols + c);
    }
    *reinterpret_cast<uint4*>(&tile[rr][ch * 8]) = v;
  }
  __syncthreads();
  const int c = c0 + threadIdx.x;
  if (c >= cols) return;
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __bfloat162float(tile[i][threadIdx.x]);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const int e = mx_scale_exponent(amax);
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i] * inv, f[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i + 2] * inv, f[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
    out[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  uint8_t* dst = codes + (static_cast<int64_t>(b) * cols + c) * ld_codes + jb * 32;   // 32-byte aligned
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(out[0]), "r"(out[1]),
               "r"(out[2]), "r"(out[3]), "r"(out[4]), "r"(out[5]), "r"(out[6]), "r"(out[7])
               : "memory");
  scales[(static_cast<int64_t>(b) * (ld_codes / 32) + jb) * ld_s + c] = static_cast<uint8_t>(e + 127);
}

// One CTA per 128 x 128 tile: thread t owns row t/2, columns (t%2)*64..+63.
__global__ void __launch_bounds__(256) fp8_tile_quant_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows,
                                                             int64_t cols, uint8_t* __restrict__ codes,
                                                             float* __restrict__ scales) {
  __shared__ float s_max[8];
  const int64_t tr = blockIdx.y, tc = blockIdx.x, b = blockIdx.z;
  const int64_t ntr = gridDim.y, ntc = gridDim.x;
  const int64_t r = tr * 128 + (threadIdx.x >> 1);
  const int64_t c0 = tc * 128 + (threadIdx.x & 1) * 64;
  const __nv_bfloat16* m = src + b * rows * cols;
  float v[64];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const int64_t c = c0 + i;
    v[i] = (r < rows && c < cols) ? __bfloat162float(m[r * cols + c]) : 0.0f;
    amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  float tmax = 0.0f;
  for (int w = 0; w < 8; ++w) tmax = fmaxf(tmax, s_max[w]);
  const float sc = tmax > 0.0f ? tmax / 448.0f : 1.0f;
  if (threadIdx.x == 0) scales[(b * ntr + tr) * ntc + tc] = sc;
  if (r >= rows) return;
  const double dsc = static_cast<double>(sc);
  uint8_t* dst = codes + b * rows * cols + r * cols;
  for (int i = 0; i < 64; ++i) {
    const int64_t c = c0 + i;
    if (c < cols)
      dst[c] = static_cast<uint8_t>(
          __nv_cvt_double_to_fp8(static_cast<double>(v[i]) / dsc, __NV_SATFINITE, __NV_E4M3));
  }
}

// Single block: counts rounded up to 128, exclusive scan over n_groups <= 1024.
__global__ void __launch_bounds__(1024) pad_offsets_kernel(const int32_t* __restrict__ offsets, int n_groups,
                                                           int32_t* __restrict__ pad_offsets) {
  __shared__ int32_t s[1024];
  const int g = threadIdx.x;
  const int32_t v = g < n_groups ? (offsets[g + 1] - offsets[g] + 127) / 128 * 128 : 0;
  s[g] = v;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    const int32_t add = g >= d ? s[g - d] : 0;
    __syncthreads();
    s[g] += add;
    __syncthreads();
  }
  if (g < n_groups) pad_offsets[g + 1] = s[g];
  if (g == 0) pad_offsets[0] = 0;
}

}  // namespace

cudaError_t launch_mx_quant_cols_t(const void* src, int64_t batch, int64_t rows, int cols,
                                   const int32_t* src_row_of, int src_div, const int32_t* offsets,
                                   const int32_t* pad_offsets, int n_groups, int64_t ld_codes, uint8_t* codes,
                                   int64_t ld_s, uint8_t* scales, cudaStream_t st) {
  if (rows <= 0 || batch <= 0) return cudaSuccess;
  if (cols <= 0 || cols % 8 || ld_codes % 32 || ld_s < cols ||
      (offsets && (!pad_offsets || batch != 1 || n_groups < 1)))
    return cudaErrorInvalidValue;
  // 16-byte source rows and 32-byte code runs
  if ((reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(codes) & 31)) return cudaErrorInvalidValue;
  if (!offsets && ld_codes < (rows + 31) / 32 * 32) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ld_codes / 32), static_cast<unsigned>((cols + 127) / 128),
                  static_cast<unsigned>(batch));
  mx_quant_cols_t_kernel<<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(src), rows, cols, src_row_of,
                                                src_div, offsets, pad_offsets, n_groups, ld_codes, codes, ld_s,
                                                scales);
  return cudaGetLastError();
}

cudaError_t launch_fp8_tile_quant(const void* src, int64_t batch, int64_t rows, int64_t cols, uint8_t* codes,
                                  float* scales, cudaStream_t st) {
  if (batch <= 0 || rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>((rows + 127) / 128),
                  static_cast<unsigned>(batch));
  fp8_tile_quant_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), rows, cols, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_pad_offsets(const int32_t* offsets, int n_groups, int32_t* pad_offsets, cudaStream_t st) {
  if (n_groups < 1 || n_groups > 1024) return cudaErrorInvalidValue;
  pad_offsets_kernel<<<1, 1024, 0, st>>>(offsets, n_groups, pad_offsets);
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_rows(const void* src, const int32_t* src_row_of, int src_div, int64_t rows, int cols,
                                 int64_t rows_per_group, int64_t ld_s, uint8_t* codes, uint8_t* scales,
                                 cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (cols % 32 || rows_per_group <= 0 || rows % rows_per_group || ld_s < rows_per_group) return cudaErrorInvalidValue;
  const int64_t warps = rows * ((cols / 32 + 31) / 32);
  const int64_t blocks = (warps + 7) / 8;
  mx_quant_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(src), src_row_of, src_div, rows, cols, rows_per_group, ld_s, codes, scales);
  return cudaGetLastError();
}

}  // namespace moe
