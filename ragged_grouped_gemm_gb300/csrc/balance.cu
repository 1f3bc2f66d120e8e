// Load-balancing side path of the router: the auxiliary loss and its logit
// gradient ("LLM Infrastructure Engineering 08: MoE Training Engineering"
// §6.2) and the load monitor statistics (§13.9).
//
// aux = coef * E * sum_i f_i P_i with f_i = counts_i / N (mean of the top-K
// mask) and P_i = mean over tokens of q_{t,i}: the softmax over all experts
// (softmax gate) or the sigmoid scores normalised over all experts (sigmoid
// gate).  Gradient with f fixed:
//   softmax: d aux / d l_{t,j} = coef * E/N * q_{t,j} (f_j - sum_i f_i q_{t,i})
//   sigmoid: d aux / d l_{t,j} = coef * E/N * s_j (1 - s_j) / S_t (f_j - sum_i f_i q_{t,i})
// Every sum runs in a fixed order (per-block partials, then one block), so
// the results do not depend on scheduling.
#include "balance.cuh"

#include <cmath>

namespace moe {
namespace {

constexpr int kTokPerBlock = 64;   // tokens of one partial row
constexpr int kMaxE = 1024;
constexpr int kPerLane = kMaxE / 32;

// q_{t,e} for e = lane + 32 j (j < nper) into q[], plus the per-token
// normaliser; returns via dq[] the factor dq_e (q_e for softmax,
// s_e (1 - s_e) / S for sigmoid).
__device__ __forceinline__ void token_probs(const float* __restrict__ row, int E, int gate, int lane,
                                            float (&q)[kPerLane], float (&dq)[kPerLane]) {
  const int nper = (E + 31) / 32;
  float v[kPerLane];
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    v[j] = (j < nper && e < E) ? row[e] : -INFINITY;
  }
  if (gate == 0) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) m = fmaxf(m, v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      v[j] = (j < nper && lane + 32 * j < E) ? expf(v[j] - m) : 0.0f;
      s += v[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.0f / s;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      q[j] = v[j] * inv;
      dq[j] = q[j];
    }
  } else {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      v[j] = (j < nper && lane + 32 * j < E) ? 1.0f / (1.0f + expf(-v[j])) : 0.0f;
      s += v[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.0f / s;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      q[j] = v[j] * inv;
      dq[j] = v[j] * (1.0f - v[j]) * inv;
    }
  }
}

// partial[b][e] = sum over the block's tokens of q_{t,e}: a warp per token
// (8 warps x 8 tokens), lane sums in registers, warps combined in warp order.
__global__ void __launch_bounds__(256) aux_partial_kernel(const float* __restrict__ logits, int N, int E, int gate,
                                                          float* __restrict__ partial) {
  __shared__ float s_acc[8][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTokPerBlock;
  float acc[kPerLane];
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) acc[j] = 0.0f;
  for (int i = warp; i < kTokPerBlock; i += 8) {
    const int t = t0 + i;
    if (t >= N) break;
    float q[kPerLane], dq[kPerLane];
    token_probs(logits + static_cast<int64_t>(t) * E, E, gate, lane, q, dq);
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) acc[j] += q[j];
  }
  const int nper = (E + 31) / 32;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j)
    if (j < nper && lane + 32 * j < E) s_acc[warp][lane + 32 * j] = acc[j];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.0f;
    for (int w = 0; w < 8; ++w) s += s_acc[w][e];
    partial[static_cast<int64_t>(blockIdx.x) * E + e] = s;
  }
}

// loss = coef * E * sum_e (counts_e / N) (sum_b partial[b][e]) / N
__global__ void __launch_bounds__(1024) aux_reduce_kernel(const float* __restrict__ partial, int nblk, int N, int E,
                                                          const int32_t* __restrict__ counts, float coef,
                                                          float* __restrict__ loss) {
  __shared__ double s_red[1024];
  const int e = threadIdx.x;
  double term = 0.0;
  if (e < E) {
    float p = 0.0f;
    for (int b = 0; b < nblk; ++b) p += partial[static_cast<int64_t>(b) * E + e];
    term = (static_cast<double>(counts[e]) / N) * (static_cast<double>(p) / N);
  }
  s_red[e] = term;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if (e < s) s_red[e] += s_red[e + s];
    __syncthreads();
  }
  if (e == 0) *loss = static_cast<float>(static_cast<double>(coef) * E * s_red[0]);
}

// dlogits_aux[t][e]: a warp per token.
__global__ void __launch_bounds__(256) aux_grad_kernel(const float* __restrict__ logits, int N, int E, int gate,
                                                       const int32_t* __restrict__ counts, float coef,
                                                       float* __restrict__ dl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= N) return;
  float q[kPerLane], dq[kPerLane];
  token_probs(logits + static_cast<int64_t>(t) * E, E, gate, lane, q, dq);
  const int nper = (E + 31) / 32;
  const float invn = 1.0f / static_cast<float>(N);
  float f[kPerLane];
  float inner = 0.0f;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    f[j] = (j < nper && e < E) ? static_cast<float>(counts[e]) * invn : 0.0f;
    inner += f[j] * q[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) inner += __shfl_xor_sync(0xffffffffu, inner, o);
  const float scale = coef * static_cast<float>(E) * invn;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    if (j < nper && e < E) dl[static_cast<int64_t>(t) * E + e] = scale * dq[j] * (f[j] - inner);
  }
}

// Monitor: the load fraction of every step in the window (counts / their
// sum, fp32 as the layer's load statistic), averaged over the steps in fp64;
// then the minimum, the entropy -sum r log(r + 1e-9) and the number of
// experts under 0.3 / E.
__global__ void __launch_bounds__(1024) monitor_kernel(const int32_t* __restrict__ hist, int H, int E,
                                                       float* __restrict__ out) {
  __shared__ double s_red[1024];
  __shared__ long long s_tot;
  const int e = threadIdx.x;
  double mean = 0.0;
  for (int h = 0; h < H; ++h) {
    const int32_t c = e < E ? hist[static_cast<int64_t>(h) * E + e] : 0;
    s_red[e] = static_cast<double>(c);
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
      if (e < s) s_red[e] += s_red[e + s];
      __syncthreads();
    }
    if (e == 0) s_tot = static_cast<long long>(s_red[0]);
    __syncthreads();
    if (e < E && s_tot > 0) mean += static_cast<double>(static_cast<float>(c) / static_cast<float>(s_tot));
    __syncthreads();
  }
  mean /= H;
  // minimum
  s_red[e] = e < E ? mean : INFINITY;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if (e < s) s_red[e] = fmin(s_red[e], s_red[e + s]);
    __syncthreads();
  }
  const double mn = s_red[0];
  __syncthreads();
  // entropy
  s_red[e] = e < E ? -mean * log(mean + 1e-9) : 0.0;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if (e < s) s_red[e] += s_red[e + s];
    __syncthreads();
  }
  const double ent = s_red[0];
  __syncthreads();
  // cold experts
  s_red[e] = (e < E && mean < 0.3 / E) ? 1.0 : 0.0;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if (e < s) s_red[e] += s_red[e + s];
    __syncthreads();
  }
  if (e == 0) {
    out[0] = static_cast<float>(mn);
    out[1] = static_cast<float>(ent);
    out[2] = static_cast<float>(s_red[0]);
  }
}

}  // namespace

size_t aux_partial_floats(int n_tok, int n_exp) {
  return static_cast<size_t>((n_tok + kTokPerBlock - 1) / kTokPerBlock) * n_exp;
}

cudaError_t launch_aux_loss(const float* logits, int n_tok, int n_exp, int gate, const int32_t* counts, float coef,
                            float* partial, float* loss, float* dlogits, cudaStream_t st) {
  if (n_exp > kMaxE || n_exp < 1 || n_tok < 1) return cudaErrorInvalidValue;
  const int nblk = (n_tok + kTokPerBlock - 1) / kTokPerBlock;
  aux_partial_kernel<<<nblk, 256, 0, st>>>(logits, n_tok, n_exp, gate, partial);
  aux_reduce_kernel<<<1, 1024, 0, st>>>(partial, nblk, n_tok, n_exp, counts, coef, loss);
  if (dlogits) aux_grad_kernel<<<(n_tok + 7) / 8, 256, 0, st>>>(logits, n_tok, n_exp, gate, counts, coef, dlogits);
  return cudaGetLastError();
}

cudaError_t launch_monitor(const int32_t* hist, int n_hist, int n_exp, float* out, cudaStream_t st) {
  if (n_exp > kMaxE || n_exp < 1 || n_hist < 1) return cudaErrorInvalidValue;
  monitor_kernel<<<1, 1024, 0, st>>>(hist, n_hist, n_exp, out);
  return cudaGetLastError();
}

}  // namespace moe
