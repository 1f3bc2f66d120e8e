// Kernel timing: CUDA events around the library's grouped-GEMM launches,
// summed per kind (moe_timing_* in moe.h; see timing.cu).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Kinds (the MOE_TIMING_* constants of moe.h).
enum TimingKind : int { TIMING_GATE = 0, TIMING_FFN_FWD = 1, TIMING_DGRAD = 2, TIMING_WGRAD = 3, TIMING_KINDS = 4 };

// Records the opening event of one timed launch on `st` and returns its slot,
// or -1 when timing is off, the pool is full or `st` is capturing a graph.
int timing_begin(int kind, cudaStream_t st);
// Records the closing event of slot `slot` (no-op for -1).
void timing_end(int slot, cudaStream_t st);

// Runs `launch` (returning cudaError_t) between the two events of one slot.
template <class F>
cudaError_t timed(int kind, cudaStream_t st, F&& launch) {
  const int slot = timing_begin(kind, st);
  const cudaError_t e = launch();
  timing_end(slot, st);
  return e;
}

}  // namespace moe
