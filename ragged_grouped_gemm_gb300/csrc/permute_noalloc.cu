// moe_permute_noalloc: the dispatch permutation for callers that cannot
// hand the library any device memory of its own.
//
// moe_permute needs a caller-provided workspace for two small per-chunk
// tables (expert histograms of 128-token chunks and their running bases).
// Some callers cannot provide one: a plugin that a host application calls
// with nothing but its input and output buffers and no allocator handle, or
// a latency-critical loop running under a fixed, pre-reserved memory budget
// where any new allocation is forbidden (cudaMalloc can block and
// synchronise the device).  For them this file keeps those two tables in a
// fixed device array that is part of the loaded library, so the call needs
// no workspace and allocates nothing.
//
// The array holds kScratchInts int32 (512 KiB) and stays resident on every
// GPU that loads the library until the process exits.  Each table needs
// ceil(n_tok / 128) * n_exp entries, so a call is accepted while that
// product is at most kScratchInts / 2 = 65536.
#include "moe.h"

#include <cuda_runtime.h>

#include <cstdint>

#include "moe_kernels.cuh"

namespace {

constexpr int kScratchInts = 2 * 65536;

static __device__ __align__(256) int32_t g_permute_scratch[kScratchInts];

// Device address of g_permute_scratch on the current device.  In host code
// the symbol's name is only a stand-in, so the address is looked up with
// cudaGetSymbolAddress, with the caller's device current.  The lookup is
// repeated on every call (a host-side query that enqueues no device work)
// rather than cached, so the address stays right after a cudaDeviceReset or
// a re-created primary context.  The first lookup on a device may load the
// library's device code there, which is why the first call on each device
// should come before any stream capture.
cudaError_t scratch_address(int32_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<int32_t*>(p);
  return cudaSuccess;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_permute_noalloc(const moe_desc_t* d, const void* x, const int32_t* topk_idx,
                                            const int32_t* offsets, int32_t* row_of_copy, int32_t* copy_of_row,
                                            void* x_perm, void* stream) {
  // Validate the description with the library's own rules (no device work).
  const moe_status_t ds = moe_workspace_size(d, nullptr, nullptr);
  if (ds != MOE_OK) return ds;
  if (!aligned16(x) || !aligned16(x_perm) || !topk_idx || !offsets || !row_of_copy || !copy_of_row)
    return MOE_ERR_INVALID_ARG;
  if (d->n_tok == 0) return MOE_OK;
  const int64_t per_table = static_cast<int64_t>(moe::permute_num_chunks(d->n_tok)) * d->n_exp;
  if (per_table > kScratchInts / 2) return MOE_ERR_WORKSPACE;   // beyond the built-in scratch
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Both tables are rewritten in full by every call, so nothing needs clearing.
  // the token-chunked map kernels, with their two chunk tables in the array
  if (moe::launch_permute_maps(d->n_tok, d->n_exp, d->top_k, topk_idx, offsets, scratch, scratch + kScratchInts / 2,
                               row_of_copy, copy_of_row, nullptr, st, /*chunked=*/true) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_permute_rows(d->n_tok, d->d_model, d->top_k, x, row_of_copy, x_perm, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
