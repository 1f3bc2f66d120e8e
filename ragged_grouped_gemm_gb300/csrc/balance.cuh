// Load-balancing side path: auxiliary loss with its logit gradient, and load
// monitor statistics (see balance.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Scratch (floats) of launch_aux_loss: per-block partial sums of the gate probabilities.
size_t aux_partial_floats(int n_tok, int n_exp);

// loss[0] = coef * E * sum_i f_i P_i; dlogits [N,E] (nullable) = its gradient with f fixed.
cudaError_t launch_aux_loss(const float* logits, int n_tok, int n_exp, int gate, const int32_t* counts, float coef,
                            float* partial, float* loss, float* dlogits, cudaStream_t st);

// out[0..2] = min load, entropy, cold experts over the n_hist rows of counts [n_hist, n_exp].
cudaError_t launch_monitor(const int32_t* hist, int n_hist, int n_exp, float* out, cudaStream_t st);

}  // namespace moe
