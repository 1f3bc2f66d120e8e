// Kernel timing of the grouped-GEMM launches (moe_timing_enable / _read /
// _disable in moe.h): a pool of CUDA event pairs created when timing is
// enabled; each timed launch takes the next pair, records one event before
// and one after the launch on the launch's stream, and notes its kind.
// Reading waits for the closing events and sums the elapsed times per kind.
#include "timing.cuh"

#include <atomic>
#include <mutex>
#include <vector>

#include "moe.h"

namespace moe {
namespace {

struct Pool {
  std::mutex mu;
  std::atomic<bool> on{false};
  std::vector<cudaEvent_t> begin, end;
  std::vector<int> kind;
  int used = 0;
  int64_t untimed[TIMING_KINDS] = {};

  void destroy() {
    for (cudaEvent_t e : begin)
      if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : end)
      if (e) cudaEventDestroy(e);
    begin.clear();
    end.clear();
    kind.clear();
    used = 0;
    for (int64_t& u : untimed) u = 0;
  }
};

Pool& pool() {
  static Pool p;
  return p;
}

}  // namespace

int timing_begin(int k, cudaStream_t st) {
  Pool& p = pool();
  if (!p.on.load(std::memory_order_acquire)) return -1;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
  if (capturing) cudaGetLastError();
  std::lock_guard<std::mutex> g(p.mu);
  if (!p.on.load(std::memory_order_relaxed)) return -1;
  if (capturing || p.used >= static_cast<int>(p.begin.size())) {
    ++p.untimed[k];
    return -1;
  }
  const int slot = p.used++;
  p.kind[slot] = k;
  if (cudaEventRecord(p.begin[slot], st) != cudaSuccess) {
    cudaGetLastError();
    p.kind[slot] = -1;   // read skips it
    ++p.untimed[k];
    return -1;
  }
  return slot;
}

void timing_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  Pool& p = pool();
  std::lock_guard<std::mutex> g(p.mu);
  if (slot >= p.used || cudaEventRecord(p.end[slot], st) != cudaSuccess) {
    cudaGetLastError();
    if (slot < p.used) {
      ++p.untimed[p.kind[slot]];
      p.kind[slot] = -1;
    }
  }
}

}  // namespace moe

extern "C" {

moe_status_t moe_timing_enable(int32_t capacity) {
  if (capacity < 1 || capacity > (1 << 20)) return MOE_ERR_INVALID_ARG;
  moe::Pool& p = moe::pool();
  std::lock_guard<std::mutex> g(p.mu);
  p.on.store(false, std::memory_order_release);
  p.destroy();
  p.begin.resize(capacity, nullptr);
  p.end.resize(capacity, nullptr);
  p.kind.assign(capacity, -1);
  for (int i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&p.begin[i]) != cudaSuccess || cudaEventCreate(&p.end[i]) != cudaSuccess) {
      cudaGetLastError();
      p.destroy();   // destroys the events created so far
      return MOE_ERR_CUDA;
    }
  }
  p.on.store(true, std::memory_order_release);
  return MOE_OK;
}

moe_status_t moe_timing_read(int32_t kind, double* total_ms, int64_t* launches, int64_t* untimed) {
  if (kind < 0 || kind >= moe::TIMING_KINDS || !total_ms || !launches) return MOE_ERR_INVALID_ARG;
  moe::Pool& p = moe::pool();
  std::lock_guard<std::mutex> g(p.mu);
  double sum = 0.0;
  int64_t n = 0;
  for (int i = 0; i < p.used; ++i) {
    if (p.kind[i] != kind) continue;
    if (cudaEventSynchronize(p.end[i]) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, p.begin[i], p.end[i]) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    sum += ms;
    ++n;
  }
  *total_ms = sum;
  *launches = n;
  if (untimed) *untimed = p.untimed[kind];
  return MOE_OK;
}

moe_status_t moe_timing_disable(void) {
  moe::Pool& p = moe::pool();
  std::lock_guard<std::mutex> g(p.mu);
  p.on.store(false, std::memory_order_release);
  p.destroy();
  return MOE_OK;
}

}  // extern "C"
