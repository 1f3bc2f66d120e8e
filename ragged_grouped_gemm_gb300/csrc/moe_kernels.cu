// Memory-bound kernels of the dropless MoE layer: router top-K with
// renormalised gate weights and the expert histogram, the exclusive scan of
// the histogram, the route-bias update, the stable expert-major permutation
// (maps and 16-byte vectorised row scatter), the gate-weighted combine, and
// the backward counterparts (combine backward with the router logit
// gradient, router weight gradient, unpermute-sum of the input gradient).
//
// Sources: "LLM Infrastructure Engineering 08: MoE Training Engineering"
// (quant67): §4.1 softmax top-K gate, §4.3 sigmoid gate with renormalisation,
// §6.3 bias-adjusted selection and online bias update, §9 simplified MoE
// layer (gate, loop over experts, index_add_, shared expert, load
// statistics, update_balance_bias), §12.5 sort by destination / bincount /
// unsort and K-sum.
#include "moe_kernels.cuh"
#include "mx_device.cuh"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kChunkTok = 128;  // tokens per chunk of the permute

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// Total order of the selection keys: larger value first, equal values by
// lower expert index, -0.0 == +0.0, NaN below every number.  The key 0 is
// reserved for "removed".
__device__ __forceinline__ unsigned long long make_key(float v, int e) {
  uint32_t u;
  if (v != v) {
    u = 0u;                                  // NaN: lowest
  } else {
    if (v == 0.0f) v = 0.0f;                 // -0.0 -> +0.0
    u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// ------------------------------------------------------------------ top-K
// Selection of one token by one warp: expert e's logit lives in lane e % 32,
// slot e / 32 of lg.  On return lanes k < K hold the k-th selected expert
// (largest key logit + bias first, the total order of make_key) and its
// renormalised gate weight: softmax over all E in fp32 then p_sel / sum
// p_sel (gate 0), or sigmoid of the unbiased logit / sum (gate 1).
template <int PL>
__device__ __forceinline__ void topk_token(const float (&lg)[PL], const float* __restrict__ bias, int E, int K,
                                           int gate, int lane, int& my_e, float& my_w) {
  unsigned long long key[PL];
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      const float kv = bias ? __fadd_rn(lg[j], bias[e]) : lg[j];
      key[j] = make_key(kv, e);
    } else {
      key[j] = 0ull;
    }
  }
  my_e = -1;
  float my_l = 0.0f;
  for (int k = 0; k < K; ++k) {
    unsigned long long best = key[0];
#pragma unroll
    for (int j = 1; j < PL; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(kFull, best, o);
      best = other > best ? other : best;
    }
    const int e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));
    float le = 0.0f;
#pragma unroll
    for (int j = 0; j < PL; ++j) {
      if (lane + 32 * j == e) {
        key[j] = 0ull;
        le = lg[j];
      }
    }
    le = __shfl_sync(kFull, le, e & 31);
    if (lane == k) {
      my_e = e;
      my_l = le;
    }
  }
  float sel;
  if (gate == 0) {
    // p = softmax over all E in fp32, then p_sel / sum(p_sel)
    float m = lg[0];
#pragma unroll
    for (int j = 1; j < PL; ++j) m = fmaxf(m, lg[j]);
    m = warp_max(m);
    float z = 0.0f;
#pragma unroll
    for (int j = 0; j < PL; ++j)
      if (lane + 32 * j < E) z += expf(lg[j] - m);
    z = warp_sum(z);
    sel = (lane < K) ? expf(my_l - m) / z : 0.0f;
  } else {
    sel = (lane < K) ? 1.0f / (1.0f + expf(-my_l)) : 0.0f;
  }
  const float tot = warp_sum(sel);
  my_w = sel / tot;
}

constexpr int kTopkMaxSlices = 4;
// One warp per token; expert e lives in lane e % 32, slot e / 32.  Top-K of
// every token from the router logits' contraction slices (added in slice
// order, fp32), the logits written, and the expert histogram and its scan
// in the same launch: each CTA adds its histogram to acc (E int32, zero
// before the launch), and the CTA that takes the last ticket writes counts
// and offsets, checks the total and leaves acc and the ticket zero.
// part: ks slices [N][E] fp32 (ks == 1: the logits themselves, not rewritten).
template <int PL>
__global__ void __launch_bounds__(256) topk_scan_kernel(RouteShape s, const float* __restrict__ part, int ks,
                                                        float* __restrict__ logits, const float* __restrict__ bias,
                                                        int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                        int32_t* acc, int32_t* ticket, int32_t* status) {
  extern __shared__ int s_hist[];
  __shared__ int s_last;
  __shared__ int s_wsum[8];
  const int E = s.n_exp, K = s.top_k;
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  const int64_t ne = static_cast<int64_t>(s.n_tok) * E;
  if (t < s.n_tok) {
    // every slice of every expert of this lane loaded first (independent
    // loads), then added in slice order
    float lg[PL], ps[PL][kTopkMaxSlices - 1];
    const float* row = part + static_cast<int64_t>(t) * E;
#pragma unroll
    for (int j = 0; j < PL; ++j) {
      const int e = lane + 32 * j;
      lg[j] = e < E ? row[e] : -INFINITY;
#pragma unroll
      for (int sl = 1; sl < kTopkMaxSlices; ++sl) ps[j][sl - 1] = (e < E && sl < ks) ? row[sl * ne + e] : 0.0f;
    }
    if (ks > 1) {
#pragma unroll
      for (int j = 0; j < PL; ++j) {
        const int e = lane + 32 * j;
#pragma unroll
        for (int sl = 1; sl < kTopkMaxSlices; ++sl)
          if (sl < ks) lg[j] += ps[j][sl - 1];
        if (e < E) logits[static_cast<int64_t>(t) * E + e] = lg[j];
      }
    }
    int my_e;
    float my_w;
    topk_token<PL>(lg, bias, E, K, s.gate, lane, my_e, my_w);
    if (lane < K) {
      topk_idx[static_cast<int64_t>(t) * K + lane] = my_e;
      topk_w[static_cast<int64_t>(t) * K + lane] = my_w;
      atomicAdd(&s_hist[my_e], 1);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (s_hist[i]) atomicAdd(acc + i, s_hist[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA: exclusive scan of the totals, four experts per thread
  int v[4], sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * threadIdx.x + j;
    v[j] = e < E ? atomicExch(acc + e, 0) : 0;
    sum += v[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += s_wsum[w];
  int run = base + incl - sum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * threadIdx.x + j;
    if (e < E) {
      counts[e] = v[j];
      run += v[j];
      offsets[e + 1] = run;
    }
  }
  if (threadIdx.x == 0) {
    offsets[0] = 0;
    *ticket = 0;
    int total = 0;
    for (int w = 0; w < 8; ++w) total += s_wsum[w];
    if (static_cast<long long>(total) != static_cast<long long>(s.n_tok) * K && status)
      atomicOr(status, DEV_BAD_OFFSETS);
  }
}

// ------------------------------------------------------------ fused router (E <= 32)
// The whole router of a layer with at most 32 experts in one launch: logits,
// top-K with renormalised weights, the expert histogram and its scan.
//
// The logits x W_g^T are a skinny contraction (N x D times D x E, E <= 32)
// bound by the read of x, so they run on the warp-level tensor-core MMA
// (mma.sync m16n8k16, bf16 in, fp32 accumulate) straight from registers:
// each CTA takes a tile of 16 tokens, its 16 warps each a contiguous
// sixteenth of the contraction, and every lane loads 16 bytes of a token row
// and of the matching W_g row per 32-column block, four blocks' loads in
// flight at once.  The contraction order inside a
// block is a fixed permutation of the columns (the same on both operands),
// and the warps' partial products are added in warp order, so the result
// is deterministic.  A warp per token then selects the top K; each CTA adds
// its expert histogram to an integer accumulator in the workspace (exact in
// any order), and the last CTA to finish (a ticket counter, no waiting)
// takes the accumulator (resetting it to zero), writes counts and offsets,
// checks that they sum to N*K, and resets the ticket.
constexpr int kRtTok = 16;
constexpr int kRtWarps = 16;
constexpr int kRtUnroll = 4;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Routing of one tile of at most 16 tokens [tok0, tok_end) by a CTA of
// kRtWarps warps: logits (each warp a slice of the contraction on the
// warp-level MMA, the slices added in warp order), then a warp per token:
// top-K, weights, and the tile's histogram in s_hist (which the caller
// zeroes).  EP = 8 * NT columns of s_acc.
template <int NT>
__device__ __forceinline__ void route_tile(const RouteShape& s, int d8, const uint4* __restrict__ x,
                                           const uint4* __restrict__ wg, const float* __restrict__ bias,
                                           float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                                           float* __restrict__ topk_w, int tok0, int tok_end,
                                           float (*s_acc)[kRtTok][8 * NT + 1], int* s_hist) {
  const int E = s.n_exp, K = s.top_k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  // this warp's 32-column blocks of the contraction
  const int nblk = d8 / 4;
  const int b0 = nblk * warp / kRtWarps, b1 = nblk * (warp + 1) / kRtWarps;
  const int r0 = tok0 + g, r1 = tok0 + g + 8;
  const bool v0 = r0 < tok_end, v1 = r1 < tok_end;
  const uint4* x0 = x + static_cast<int64_t>(v0 ? r0 : 0) * d8 + q;
  const uint4* x1 = x + static_cast<int64_t>(v1 ? r1 : 0) * d8 + q;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  float c[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
  for (int b = b0; b < b1; b += kRtUnroll) {
    uint4 xa[kRtUnroll], xb[kRtUnroll], w[kRtUnroll][NT];
#pragma unroll
    for (int u = 0; u < kRtUnroll; ++u) {
      const bool in = b + u < b1;
      xa[u] = (in && v0) ? ld_stream(x0 + 4 * (b + u)) : zero;
      xb[u] = (in && v1) ? ld_stream(x1 + 4 * (b + u)) : zero;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int e = 8 * j + g;
        w[u][j] = (in && e < E) ? __ldg(wg + static_cast<int64_t>(e) * d8 + 4 * (b + u) + q) : zero;
      }
    }
#pragma unroll
    for (int u = 0; u < kRtUnroll; ++u) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        // lane (g, q) holds columns 8q..8q+7 of rows g, g+8 and of W_g row 8j+g:
        // columns 8q+0..3 form the first k16 step, 8q+4..7 the second
        mma_bf16_16816(c[j], xa[u].x, xb[u].x, xa[u].y, xb[u].y, w[u][j].x, w[u][j].y);
        mma_bf16_16816(c[j], xa[u].z, xb[u].z, xa[u].w, xb[u].w, w[u][j].z, w[u][j].w);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    s_acc[warp][g][8 * j + 2 * q] = c[j][0];
    s_acc[warp][g][8 * j + 2 * q + 1] = c[j][1];
    s_acc[warp][g + 8][8 * j + 2 * q] = c[j][2];
    s_acc[warp][g + 8][8 * j + 2 * q + 1] = c[j][3];
  }
  __syncthreads();
  // a token per warp: logits (partials added in warp order), top-K, weights
  for (int tt = warp; tt < kRtTok; tt += kRtWarps) {
    const int t = tok0 + tt;
    if (t >= tok_end) break;
    float lg[1];
    float v = 0.0f;
    if (lane < E) {
#pragma unroll
      for (int w = 0; w < kRtWarps; ++w) v += s_acc[w][tt][lane];
      logits[static_cast<int64_t>(t) * E + lane] = v;
    }
    lg[0] = lane < E ? v : -INFINITY;
    int my_e;
    float my_w;
    topk_token<1>(lg, bias, E, K, s.gate, lane, my_e, my_w);
    if (lane < K) {
      topk_idx[static_cast<int64_t>(t) * K + lane] = my_e;
      topk_w[static_cast<int64_t>(t) * K + lane] = my_w;
      atomicAdd(&s_hist[my_e], 1);
    }
  }
}

template <int NT>   // 8-expert column tiles: E <= 8 * NT
__global__ void __launch_bounds__(kRtWarps * 32) router_fused_kernel(
    RouteShape s, int d8, const uint4* __restrict__ x, const uint4* __restrict__ wg, const float* __restrict__ bias,
    float* __restrict__ logits, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* acc, int32_t* ticket, int32_t* status) {
  constexpr int EP = 8 * NT;
  __shared__ float s_acc[kRtWarps][kRtTok][EP + 1];
  __shared__ int s_hist[32];
  __shared__ int s_last;
  const int E = s.n_exp, K = s.top_k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 32) s_hist[threadIdx.x] = 0;
  __syncthreads();
  route_tile<NT>(s, d8, x, wg, bias, logits, topk_idx, topk_w, blockIdx.x * kRtTok,
                 min(s.n_tok, static_cast<int>(blockIdx.x + 1) * kRtTok), s_acc, s_hist);
  __syncthreads();
  if (threadIdx.x < E && s_hist[threadIdx.x]) atomicAdd(acc + threadIdx.x, s_hist[threadIdx.x]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA: every CTA's histogram is in the accumulator; take it, then its scan
  if (warp == 0) {
    const int tot = lane < E ? atomicExch(acc + lane, 0) : 0;
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane < E) {
      counts[lane] = tot;
      offsets[lane + 1] = incl;
    }
    if (lane == 0) {
      offsets[0] = 0;
      *ticket = 0;
    }
    const int total = __shfl_sync(kFull, incl, E - 1);
    if (lane == 0 && static_cast<long long>(total) != static_cast<long long>(s.n_tok) * K && status)
      atomicOr(status, DEV_BAD_OFFSETS);
  }
}

// ------------------------------------------------------------ route + permute
// moe_route followed by moe_permute in one cooperative launch (E <= 32).
// Phase 1: each CTA routes its 16-token tiles (route_tile) and publishes each
// tile's expert histogram th[tile][E].  A bounded grid-wide barrier follows
// (the launch is cooperative, so every CTA is resident).  Phase 2: each CTA
// adds up the histograms - the experts' totals give counts and offsets, the
// tiles before each of its own give that tile's first row per expert - then
// assigns its copies' rows in copy order (as the permute kernels do) and
// copies its token rows, which phase 1 has just read (so they come from L2).
// bar: arrivals in bar[0] and the generation in bar[32] (another 128-byte
// line, so the waiting CTAs' polls do not contend with the arrivals), zero
// after moe_workspace_init; the last CTA to arrive resets the arrivals.
__device__ __forceinline__ bool grid_barrier_bounded(int32_t* bar, int32_t* status, int site) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_ok = 1;
    volatile int32_t* vgen = bar + 32;
    const int32_t gen = *vgen;
    __threadfence();
    if (atomicAdd(bar, 1) == static_cast<int>(gridDim.x) - 1) {
      bar[0] = 0;
      __threadfence();
      atomicAdd(bar + 32, 1);
    } else {
      const uint64_t t0 = globaltimer_ns();
      uint32_t n = 0;
      while (*vgen == gen) {
        __nanosleep(32);
        if ((++n & 63u) == 0 && globaltimer_ns() - t0 > kSpinTimeoutNs) {
          s_ok = 0;
          if (status) {
            atomicOr(status, DEV_TIMEOUT);
            atomicExch(status + 1, site);
          }
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  return s_ok != 0;
}

constexpr int kRpCopyBatch = 8;   // token rows a thread's copy loads keep in flight

// Of T tiles, the first N mod T hold q + 1 tokens and the rest q, q = N / T
// (at most 16 each, in token order); T is a multiple of the grid where that
// balances the CTAs.  Tile t starts at token t*q + min(t, N mod T).
__device__ __forceinline__ int rp_tile_begin(int t, int q, int rem) { return t * q + min(t, rem); }

// Per expert, the sum of th[t][e] over tiles t < t_mid (into pre) and over
// t_mid <= t < t_hi (into post), both zeroed by the caller: the CTA's threads
// each take entries j = tid, tid + blockDim, ... of th[t_lo..t_hi) (all their
// loads in flight at once) and add them with shared-memory atomics.
__device__ __forceinline__ void rp_hist_sums(const int32_t* th, int E, int t_lo, int t_mid, int t_hi, int* pre,
                                             int* post) {
  constexpr int kLoads = 4;
  const int n = (t_hi - t_lo) * E;   // at most (ceil(N/16) + 2048) * 32 entries
  const int split = (t_mid - t_lo) * E;
  const int32_t* src = th + static_cast<int64_t>(t_lo) * E;
  for (int j0 = threadIdx.x; j0 < n; j0 += kLoads * blockDim.x) {
    int v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int j = j0 + u * blockDim.x;
      v[u] = j < n ? __ldcg(src + j) : 0;
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int j = j0 + u * blockDim.x;
      if (j < n && v[u]) atomicAdd(j < split ? &pre[j % E] : &post[j % E], v[u]);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kRtWarps * 32, 2) route_permute_kernel(
    RouteShape s, int d8, int ntiles, int tq, int trem, const uint4* __restrict__ x, const uint4* __restrict__ wg,
    const float* __restrict__ bias, float* __restrict__ logits, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_of_copy, int32_t* __restrict__ copy_of_row, uint4* __restrict__ x_perm, int32_t* th,
    int32_t* bar, int32_t* status) {
  constexpr int EP = 8 * NT;
  __shared__ float s_acc[kRtWarps][kRtTok][EP + 1];
  __shared__ int s_hist[32];
  __shared__ int s_off[33];
  __shared__ int s_pre[32];
  __shared__ int s_post[32];
  __shared__ int s_base[32];
  __shared__ int s_pos[kRtTok * 32];
  __shared__ int s_bad;
  const int E = s.n_exp, K = s.top_k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t R = static_cast<int64_t>(s.n_tok) * K;
  if (tid == 0) s_bad = 0;
  // ---- phase 1: routing
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    if (tid < 32) s_hist[tid] = 0;
    __syncthreads();
    route_tile<NT>(s, d8, x, wg, bias, logits, topk_idx, topk_w, rp_tile_begin(tile, tq, trem),
                   rp_tile_begin(tile + 1, tq, trem), s_acc, s_hist);
    __syncthreads();
    if (tid < E) {
      th[static_cast<int64_t>(tile) * E + tid] = s_hist[tid];
      __threadfence();   // each writer orders its histogram word before the barrier's arrival
    }
  }
  if (tid < 32) {
    s_pre[tid] = 0;
    s_post[tid] = 0;
  }
  if (!grid_barrier_bounded(bar, status, 710)) return;
  // ---- phase 2: the experts' totals and the tiles before this CTA's first
  // tile, in one pass over the histograms
  rp_hist_sums(th, E, 0, blockIdx.x, ntiles, s_pre, s_post);
  __syncthreads();
  if (warp == 0) {
    int pre = s_pre[lane], tot = pre + s_post[lane];
    if (lane >= E) tot = pre = 0;
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    s_off[lane + 1] = incl;
    if (lane == 0) s_off[0] = 0;
    s_pre[lane] = pre;
    if (blockIdx.x == 0) {
      if (lane < E) {
        counts[lane] = tot;
        offsets[lane + 1] = incl;
      }
      if (lane == 0) offsets[0] = 0;
      const int total = __shfl_sync(kFull, incl, 31);
      if (lane == 0 && static_cast<long long>(total) != R && status) atomicOr(status, DEV_BAD_OFFSETS);
    }
  }
  __syncthreads();
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    // this tile's first row per expert: offsets plus the copies of the tiles
    // before it (the running prefix gains the tiles since this CTA's last one)
    if (tile != static_cast<int>(blockIdx.x)) {
      rp_hist_sums(th, E, tile - static_cast<int>(gridDim.x), tile, tile, s_pre, s_post);
    }
    __syncthreads();
    if (warp == 0) s_base[lane] = s_off[lane] + s_pre[lane];
    __syncthreads();
    // rows of the tile's copies in copy order (warp 0)
    const int t0k = rp_tile_begin(tile, tq, trem);
    const int ntk = rp_tile_begin(tile + 1, tq, trem) - t0k;
    const int64_t c0 = static_cast<int64_t>(t0k) * K;
    const int ncp = ntk * K;
    if (warp == 0) {
      for (int b = 0; b < ncp; b += 32) {
        const int i = b + lane;
        const bool active = i < ncp;
        const int e = active ? __ldcg(topk_idx + c0 + i) : -1;
        const bool ok = active && e >= 0 && e < E;
        const unsigned am = __ballot_sync(kFull, ok);
        int pos = -1;
        if (ok) {
          const unsigned m = __match_any_sync(am, e);
          const int leader = __ffs(m) - 1;
          const int rank = __popc(m & ((1u << lane) - 1u));
          int base = 0;
          if (lane == leader) {
            base = s_base[e];
            s_base[e] = base + __popc(m);
          }
          base = __shfl_sync(am, base, leader);
          pos = base + rank;
          if (!(pos >= 0 && pos < s_off[e + 1] && pos < R)) {
            pos = -1;
            atomicOr(&s_bad, DEV_BAD_OFFSETS);
          }
        } else if (active) {
          atomicOr(&s_bad, DEV_BAD_INDEX);
        }
        if (active) {
          s_pos[i] = pos;
          row_of_copy[c0 + i] = pos;
          if (pos >= 0) copy_of_row[pos] = static_cast<int32_t>(c0 + i);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    // the tile's token rows (read by phase 1, so from L2), each read once and
    // written to its copies' rows
    for (int i = tid; i < d8; i += kRtWarps * 32) {
#pragma unroll
      for (int tb = 0; tb < kRtTok; tb += kRpCopyBatch) {
        uint4 v[kRpCopyBatch];
#pragma unroll
        for (int u = 0; u < kRpCopyBatch; ++u)
          v[u] = tb + u < ntk ? x[static_cast<int64_t>(t0k + tb + u) * d8 + i] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kRpCopyBatch; ++u) {
          if (tb + u >= ntk) break;
          for (int k = 0; k < K; ++k) {
            const int r = s_pos[(tb + u) * K + k];
            if (r >= 0) x_perm[static_cast<int64_t>(r) * d8 + i] = v[u];
          }
        }
      }
    }
    __syncthreads();
  }
  if (tid == 0 && s_bad && status) atomicOr(status, s_bad);
}

// ------------------------------------------------------------ bias update
__global__ void update_bias_kernel(const int32_t* __restrict__ counts, int E, float* __restrict__ bias, float gamma,
                                   int mode, float target) {
  __shared__ long long s_total;
  if (threadIdx.x == 0) {
    long long tot = 0;
    for (int e = 0; e < E; ++e) tot += counts[e];
    s_total = tot;
  }
  __syncthreads();
  if (s_total == 0) return;  // empty batch: leave the bias unchanged
  const float total = static_cast<float>(s_total);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float ls = __fdiv_rn(static_cast<float>(counts[e]), total);
    const float diff = __fsub_rn(ls, target);
    const float sgn = diff > 0.0f ? 1.0f : (diff < 0.0f ? -1.0f : 0.0f);
    float step = __fmul_rn(gamma, sgn);
    if (mode == 0) step = __fmul_rn(step, fmaxf(ls, 1e-6f));
    bias[e] = __fsub_rn(bias[e], step);
  }
}

// ------------------------------------------------------------ permutation
__global__ void __launch_bounds__(256) block_hist_kernel(int n_tok, int E, int K, const int32_t* __restrict__ idx,
                                                         int32_t* __restrict__ block_counts, int32_t* status) {
  extern __shared__ int s_h[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_h[i] = 0;
  __syncthreads();
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunkTok * K;
  const int64_t c1 = min(static_cast<int64_t>(n_tok) * K, c0 + static_cast<int64_t>(kChunkTok) * K);
  for (int64_t c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
    const int e = idx[c];
    if (e >= 0 && e < E) atomicAdd(&s_h[e], 1);
    else if (status) atomicOr(status, DEV_BAD_INDEX);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    block_counts[static_cast<int64_t>(blockIdx.x) * E + i] = s_h[i];
}

// Each expert's first row per chunk.  The caller's offsets must be the
// exclusive scan of the histogram; an expert whose rows do not end at
// offsets[e+1] is reported as DEV_BAD_OFFSETS (the scatter then drops the
// copies that fall outside [offsets[e], offsets[e+1]) or [0, R)).
__global__ void block_base_kernel(int nchunks, int E, const int32_t* __restrict__ offsets,
                                  const int32_t* __restrict__ block_counts, int32_t* __restrict__ block_base,
                                  int32_t* status) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  int run = offsets[e];
  for (int ch = 0; ch < nchunks; ++ch) {
    block_base[static_cast<int64_t>(ch) * E + e] = run;
    run += block_counts[static_cast<int64_t>(ch) * E + e];
  }
  if (run != offsets[e + 1] && status) atomicOr(status, DEV_BAD_OFFSETS);
}

// One warp per chunk of tokens; copies are visited in copy order c = t*K+k,
// (32/K) tokens per step, so each expert's rows come out in ascending token
// order (ties of a repeated expert inside one token by ascending k).
// A position outside the expert's own rows [offsets[e], offsets[e+1]) or
// outside [0, R) (offsets inconsistent with the expert indices) is not
// written: the copy gets row -1 and DEV_BAD_OFFSETS is raised.
__global__ void __launch_bounds__(32) scatter_maps_kernel(int n_tok, int E, int K, const int32_t* __restrict__ idx,
                                                          const int32_t* __restrict__ offsets,
                                                          const int32_t* __restrict__ block_base,
                                                          int32_t* __restrict__ row_of_copy,
                                                          int32_t* __restrict__ copy_of_row, int32_t* status) {
  extern __shared__ int s_base[];
  int* s_end = s_base + E;
  const int lane = threadIdx.x;
  const int64_t R = static_cast<int64_t>(n_tok) * K;
  for (int i = lane; i < E; i += 32) {
    s_base[i] = block_base[static_cast<int64_t>(blockIdx.x) * E + i];
    s_end[i] = offsets[i + 1];
  }
  __syncwarp();
  const int t_begin = blockIdx.x * kChunkTok;
  const int t_end = min(n_tok, t_begin + kChunkTok);
  const int tpi = 32 / K;
  for (int t0 = t_begin; t0 < t_end; t0 += tpi) {
    const int t = t0 + lane / K;
    const int k = lane - (lane / K) * K;
    const bool active = (lane < tpi * K) && (t < t_end);
    const int64_t c = static_cast<int64_t>(t) * K + k;
    const int e = active ? idx[c] : -1;
    const bool ok = active && e >= 0 && e < E;
    const unsigned am = __ballot_sync(kFull, ok);
    if (ok) {
      const unsigned m = __match_any_sync(am, e);
      const int leader = __ffs(m) - 1;
      const int rank = __popc(m & ((1u << lane) - 1u));
      int base = 0;
      if (lane == leader) {
        base = s_base[e];
        s_base[e] = base + __popc(m);
      }
      base = __shfl_sync(am, base, leader);
      const int pos = base + rank;
      if (pos >= 0 && pos < s_end[e] && pos < R) {
        row_of_copy[c] = pos;
        copy_of_row[pos] = static_cast<int32_t>(c);
      } else {
        row_of_copy[c] = -1;
        if (status) atomicOr(status, DEV_BAD_OFFSETS);
      }
    } else if (active) {
      row_of_copy[c] = -1;   // expert index outside [0, E): no row (reported by block_hist_kernel)
    }
    __syncwarp();
  }
}

// Single-CTA form of the three kernels above for up to kMapOnePassMax
// copies: the copies c = 0..R-1 are cut into 32 contiguous segments, one per
// warp; each warp counts its segment's copies per expert (warp-aggregated
// through __match_any_sync), then one thread per expert turns the 32 counts
// into the segment's first row of that expert (a running sum from
// offsets[e], checked against offsets[e+1]), and each warp walks its
// segment again in copy order assigning rows exactly as scatter_maps_kernel
// does (same positions, same bound checks, same status bits).  Each lane
// keeps kMapBatch copies' expert indices in registers per pass, so the
// segment is read with kMapBatch independent loads in flight.
constexpr int kMapBatch = 8;
constexpr int64_t kMapOnePassMax = 65536;

__global__ void __launch_bounds__(1024, 1) maps_onepass_kernel(int n_tok, int E, int K,
                                                               const int32_t* __restrict__ idx,
                                                               const int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ row_of_copy,
                                                               int32_t* __restrict__ copy_of_row, int32_t* status) {
  extern __shared__ int s_map[];
  int* s_seg = s_map;              // [32][E]: segment counts, then segment bases
  int* s_end = s_map + 32 * E;     // [E]: offsets[e + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t R = static_cast<int64_t>(n_tok) * K;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) s_seg[i] = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_end[i] = offsets[i + 1];
  __syncthreads();
  const int64_t per = (R + 31) / 32;
  const int64_t c0 = min(R, warp * per), c1 = min(R, c0 + per);
  int* hist = s_seg + warp * E;
  bool bad_index = false, bad_offsets = false;
  for (int64_t b = c0; b < c1; b += 32 * kMapBatch) {
    int e[kMapBatch];
#pragma unroll
    for (int j = 0; j < kMapBatch; ++j) {
      const int64_t c = b + 32 * j + lane;
      e[j] = c < c1 ? idx[c] : -1;
    }
#pragma unroll
    for (int j = 0; j < kMapBatch; ++j) {
      const int64_t c = b + 32 * j + lane;
      const bool active = c < c1;
      const bool ok = active && e[j] >= 0 && e[j] < E;
      bad_index |= active && !ok;
      const unsigned am = __ballot_sync(kFull, ok);
      if (ok) {
        const unsigned m = __match_any_sync(am, e[j]);
        if (lane == __ffs(m) - 1) hist[e[j]] += __popc(m);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {
    int run = offsets[ex];
    for (int w = 0; w < 32; ++w) {
      const int n = s_seg[w * E + ex];
      s_seg[w * E + ex] = run;
      run += n;
    }
    bad_offsets |= run != s_end[ex];
  }
  __syncthreads();
  for (int64_t b = c0; b < c1; b += 32 * kMapBatch) {
    int e[kMapBatch];
#pragma unroll
    for (int j = 0; j < kMapBatch; ++j) {
      const int64_t c = b + 32 * j + lane;
      e[j] = c < c1 ? idx[c] : -1;
    }
#pragma unroll
    for (int j = 0; j < kMapBatch; ++j) {
      const int64_t c = b + 32 * j + lane;
      const bool active = c < c1;
      const bool ok = active && e[j] >= 0 && e[j] < E;
      const unsigned am = __ballot_sync(kFull, ok);
      if (ok) {
        const unsigned m = __match_any_sync(am, e[j]);
        const int leader = __ffs(m) - 1;
        const int rank = __popc(m & ((1u << lane) - 1u));
        int base = 0;
        if (lane == leader) {
          base = hist[e[j]];
          hist[e[j]] = base + __popc(m);
        }
        base = __shfl_sync(am, base, leader);
        const int pos = base + rank;
        if (pos >= 0 && pos < s_end[e[j]] && pos < R) {
          row_of_copy[c] = pos;
          copy_of_row[pos] = static_cast<int32_t>(c);
        } else {
          row_of_copy[c] = -1;
          bad_offsets = true;
        }
      } else if (active) {
        row_of_copy[c] = -1;   // expert index outside [0, E): no row
      }
      __syncwarp();
    }
  }
  if (status) {
    if (bad_index) atomicOr(status, DEV_BAD_INDEX);
    if (bad_offsets) atomicOr(status, DEV_BAD_OFFSETS);
  }
}

// ------------------------------------------------------------ single-pass permute
// The whole dispatch of moe_permute in one launch: stable maps and the row
// copy.  The copies are cut into chunks of kSpTok tokens; a CTA takes the next
// chunk from a ticket counter (so every chunk before it has a CTA already
// running), counts its chunk's copies per expert, and publishes per expert a
// 64-bit word {tag (32 bits), state (1 bit), value (31 bits)}: first the
// chunk's own count (state "aggregate"), and once known its inclusive row
// prefix (state "prefix"; chunk 0 publishes offsets[e] + count at once).  A
// chunk's first row of expert e is found by walking back over the preceding
// chunks' words, adding aggregates until a prefix is met (decoupled
// look-back).  All of a CTA's threads walk at once: S = 32, 16, ... 1 lanes
// per expert so that every expert has its lanes (S * E <= kSpThreads where it
// fits), each lane with kSpLook words in flight, so one round trip covers
// S * kSpLook preceding chunks of every expert; the nearest chunk with a
// prefix ends the walk, and the values after it are added by a shuffle
// reduction over the expert's lanes.  Every wait on a word
// not yet published this call is bounded and reports MOE_DEV_TIMEOUT.
// The tag is the call's generation + 1 (the generation counter and the words
// start at zero after moe_workspace_init; the last CTA of a call advances
// the generation and resets the ticket).  The words live in a region of the
// workspace that holds nothing else, so a word is either zero or left by an
// earlier call, and never reads as this call's (until the 32-bit generation
// wraps, after 2^32 - 1 calls on one workspace).  Positions inside the chunk follow copy order,
// exactly as the other map kernels assign them, with the same bound checks;
// then the chunk's token rows are read once and written to their K rows.
constexpr int kSpTok = 16;
constexpr int kSpThreads = 256;
constexpr int kSpLook = 16;   // look-back words in flight per lane
constexpr uint64_t kSpAggregate = 0, kSpPrefix = 1;

__device__ __forceinline__ uint64_t sp_word(uint32_t tag, uint64_t state, int value) {
  return (static_cast<uint64_t>(tag) << 32) | (state << 31) | (static_cast<uint32_t>(value) & 0x7FFFFFFFu);
}

// MXFP8 outputs of the quantising form: codes [rows][d] and E8M0 scales
// [d/32][ld] of the permuted rows, and (nullable) of the token rows.
struct SpQuantOut {
  uint8_t* codes;
  uint8_t* scales;
  int64_t ld;
  uint8_t* tok_codes;
  uint8_t* tok_scales;
  int64_t tok_ld;
};

template <bool QUANT>
__global__ void __launch_bounds__(kSpThreads, 2) permute_single_pass_kernel(
    int n_tok, int E, int K, int d8, const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets,
    const uint4* __restrict__ x, int32_t* __restrict__ row_of_copy, int32_t* __restrict__ copy_of_row,
    uint4* __restrict__ x_perm, unsigned long long* look, int32_t* ctl, int32_t* status, SpQuantOut q) {
  extern __shared__ int s_sp[];
  int* s_h = s_sp;                    // [E] the chunk's copies per expert
  int* s_base = s_sp + E;             // [E] the chunk's next row per expert
  int* s_e = s_sp + 2 * E;            // [kSpTok * K] expert of each copy
  int* s_pos = s_e + kSpTok * K;      // [kSpTok * K] row of each copy (-1: none)
  __shared__ int s_chunk;
  __shared__ uint32_t s_tag;
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_chunk = atomicAdd(ctl, 1);
    s_tag = static_cast<uint32_t>(*reinterpret_cast<volatile int32_t*>(ctl + 2)) + 1u;
    s_bad = 0;
  }
  for (int e = tid; e < E; e += kSpThreads) s_h[e] = 0;
  __syncthreads();
  const int chunk = s_chunk;
  const uint32_t tag = s_tag;
  const int64_t R = static_cast<int64_t>(n_tok) * K;
  const int64_t c0 = static_cast<int64_t>(chunk) * kSpTok * K;
  const int ncp = static_cast<int>(min(R - c0, static_cast<int64_t>(kSpTok) * K));
  for (int i = tid; i < ncp; i += kSpThreads) {
    const int e = idx[c0 + i];
    s_e[i] = e;
    if (e >= 0 && e < E) atomicAdd(&s_h[e], 1);
    else atomicOr(&s_bad, DEV_BAD_INDEX);
  }
  __syncthreads();
  volatile unsigned long long* vlook = look;
  // bf16: this thread's first 16-byte column of the chunk's token rows is
  // loaded now, so the reads are in flight during the look-back
  const int t0k = chunk * kSpTok;
  const int ntk = ncp / K;
  uint4 v[kSpTok];
  if (!QUANT && tid < d8) {
#pragma unroll
    for (int tt = 0; tt < kSpTok; ++tt)
      v[tt] = tt < ntk ? x[static_cast<int64_t>(t0k + tt) * d8 + tid] : make_uint4(0, 0, 0, 0);
  }
  if (QUANT && tid < ntk * (d8 / 4)) {   // QUANT: this thread's first 32-element block
    const uint4* src = x + static_cast<int64_t>(t0k + tid / (d8 / 4)) * d8 + (tid % (d8 / 4)) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = src[j];
  }
  // publish this chunk's aggregates (chunk 0: its prefixes)
  for (int e = tid; e < E; e += kSpThreads) {
    unsigned long long* mine = look + static_cast<int64_t>(chunk) * E + e;
    if (chunk == 0) {
      s_base[e] = offsets[e];
      *reinterpret_cast<volatile unsigned long long*>(mine) = sp_word(tag, kSpPrefix, offsets[e] + s_h[e]);
    } else {
      *reinterpret_cast<volatile unsigned long long*>(mine) = sp_word(tag, kSpAggregate, s_h[e]);
    }
  }
  if (chunk > 0) {
    // look-back: S lanes per expert (a power of two; S * experts per pass =
    // kSpThreads), lane u of an expert's group reads the words of chunks
    // j0 - u - S*l, l < kSpLook, all in flight together.  The nearest chunk
    // with a prefix ends the walk; the values from it up to chunk - 1 are
    // summed over the group.
    int S = 32;
    while (S > 1 && S * E > kSpThreads) S >>= 1;
    const int per_pass = kSpThreads / S;
    const int u = tid & (S - 1);
    const unsigned gmask = S == 32 ? kFull : (((1u << S) - 1u) << (lane & ~(S - 1)));
    for (int e = tid / S; e < E; e += per_pass) {   // uniform within each group of S lanes
      int acc = 0;
      int j0 = chunk - 1;
      uint64_t t0 = 0;
      while (j0 >= 0) {
        unsigned long long w[kSpLook];
#pragma unroll
        for (int l = 0; l < kSpLook; ++l) {
          const int j = j0 - u - S * l;
          w[l] = j >= 0 ? vlook[static_cast<int64_t>(j) * E + e] : 0ull;
        }
        int jp = -1;   // this lane's nearest chunk with a prefix
#pragma unroll
        for (int l = kSpLook - 1; l >= 0; --l) {
          const int j = j0 - u - S * l;
          if (j >= 0 && static_cast<uint32_t>(w[l] >> 32) == tag && ((w[l] >> 31) & 1u) == kSpPrefix) jp = j;
        }
        for (int o = S >> 1; o; o >>= 1) jp = max(jp, __shfl_xor_sync(gmask, jp, o, S));
        int nr = 0, v = 0;   // a chunk from the prefix on that has not published yet; the sum
#pragma unroll
        for (int l = 0; l < kSpLook; ++l) {
          const int j = j0 - u - S * l;
          if (j >= 0 && j >= jp) {
            if (static_cast<uint32_t>(w[l] >> 32) != tag) nr = 1;
            else v += static_cast<int>(static_cast<uint32_t>(w[l]) & 0x7FFFFFFFu);
          }
        }
        for (int o = S >> 1; o; o >>= 1) {
          nr |= __shfl_xor_sync(gmask, nr, o, S);
          v += __shfl_xor_sync(gmask, v, o, S);
        }
        if (nr) {   // read the window again (bounded); lane 0 of the group decides for it
          int out = 0;
          if (u == 0) {
            if (t0 == 0) t0 = globaltimer_ns();
            else out = globaltimer_ns() - t0 > kSpinTimeoutNs;
          }
          if (__shfl_sync(gmask, out, 0, S)) {
            if (u == 0) {
              atomicOr(&s_bad, DEV_TIMEOUT);
              if (status) atomicExch(status + 1, 700);
            }
            break;
          }
          continue;
        }
        acc += v;
        if (jp >= 0) break;
        j0 -= S * kSpLook;
        t0 = 0;
      }
      if (u == 0) {
        s_base[e] = acc;
        *reinterpret_cast<volatile unsigned long long*>(look + static_cast<int64_t>(chunk) * E + e) =
            sp_word(tag, kSpPrefix, acc + s_h[e]);
      }
    }
  }
  __syncthreads();
  // rows of the chunk's copies in copy order (warp 0)
  if (warp == 0) {
    for (int b = 0; b < ncp; b += 32) {
      const int i = b + lane;
      const bool active = i < ncp;
      const int e = active ? s_e[i] : -1;
      const bool ok = active && e >= 0 && e < E;
      const unsigned am = __ballot_sync(kFull, ok);
      int pos = -1;
      if (ok) {
        const unsigned m = __match_any_sync(am, e);
        const int leader = __ffs(m) - 1;
        const int rank = __popc(m & ((1u << lane) - 1u));
        int base = 0;
        if (lane == leader) {
          base = s_base[e];
          s_base[e] = base + __popc(m);
        }
        base = __shfl_sync(am, base, leader);
        pos = base + rank;
        if (!(pos >= 0 && pos < offsets[e + 1] && pos < R)) {
          pos = -1;
          atomicOr(&s_bad, DEV_BAD_OFFSETS);
        }
      }
      if (active) {
        s_pos[i] = pos;
        row_of_copy[c0 + i] = pos;
        if (pos >= 0) copy_of_row[pos] = static_cast<int32_t>(c0 + i);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // the chunk's token rows, each read once and written to its copies' rows:
  // a thread takes one 16-byte column chunk of all the chunk's tokens (their
  // loads in flight together; the first chunk was loaded before the
  // look-back), then stores each to its K rows.  QUANT: a thread takes one
  // 32-element block of a token, quantises it once (the row quantiser's
  // arithmetic) and writes its codes and scale byte to the token's K rows
  // (and to the token row)
  if (QUANT) {
    const int nkb = d8 / 4;
    const int64_t d = static_cast<int64_t>(d8) * 8;    // elements per row = code bytes per row
    for (int u = tid; u < ntk * nkb; u += kSpThreads) {
      const int tt = u / nkb;
      const int kb = u - tt * nkb;
      const int64_t tok = t0k + tt;
      uint4 vb[4];
      if (u == tid) {   // loaded before the look-back
#pragma unroll
        for (int j = 0; j < 4; ++j) vb[j] = v[j];
      } else {
        const uint4* src = x + tok * d8 + kb * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) vb[j] = src[j];
      }
      uint4 c0, c1;
      const uint8_t sc = mx_quant_block32(vb, c0, c1);
      for (int k = 0; k < K; ++k) {
        const int r = s_pos[tt * K + k];
        if (r < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(q.codes + static_cast<int64_t>(r) * d + kb * 32);
        dst[0] = c0;
        dst[1] = c1;
        q.scales[static_cast<int64_t>(kb) * q.ld + r] = sc;
      }
      if (q.tok_codes) {
        uint4* dst = reinterpret_cast<uint4*>(q.tok_codes + tok * d + kb * 32);
        dst[0] = c0;
        dst[1] = c1;
        q.tok_scales[static_cast<int64_t>(kb) * q.tok_ld + tok] = sc;
      }
    }
  }
  for (int i = tid; i < (QUANT ? 0 : d8); i += kSpThreads) {
    if (i != tid) {
#pragma unroll
      for (int tt = 0; tt < kSpTok; ++tt)
        v[tt] = tt < ntk ? x[static_cast<int64_t>(t0k + tt) * d8 + i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int tt = 0; tt < kSpTok; ++tt) {
      if (tt >= ntk) break;
      for (int k = 0; k < K; ++k) {
        const int r = s_pos[tt * K + k];
        if (r >= 0) x_perm[static_cast<int64_t>(r) * d8 + i] = v[tt];
      }
    }
  }
  if (tid == 0) {
    if (s_bad && status) atomicOr(status, s_bad);
    __threadfence();
    if (atomicAdd(ctl + 1, 1) == static_cast<int>(gridDim.x) - 1) {   // last CTA: next call's state
      ctl[0] = 0;
      ctl[1] = 0;
      atomicAdd(ctl + 2, 1);
    }
  }
}

__global__ void __launch_bounds__(256) permute_rows_kernel(int n_tok, int d8, int K, const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ row_of_copy,
                                                           uint4* __restrict__ x_perm) {
  __shared__ int s_rows[32];
  for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < K) s_rows[threadIdx.x] = row_of_copy[static_cast<int64_t>(t) * K + threadIdx.x];
    __syncthreads();
    const uint4* src = x + static_cast<int64_t>(t) * d8;
    for (int i = threadIdx.x; i < d8; i += blockDim.x) {
      const uint4 v = src[i];
      for (int k = 0; k < K; ++k)
        if (s_rows[k] >= 0) x_perm[static_cast<int64_t>(s_rows[k]) * d8 + i] = v;   // -1: dropped copy
    }
  }
}

// ------------------------------------------------------------ combine
// A warp per (token, segment of 128 16-byte chunks of its row); lane l
// handles chunks l, l+32, l+64, l+96 of the segment, so every load and store
// instruction of the warp covers 512 contiguous bytes.  The K copies' rows
// are loaded NB copies at a time (4 * NB 16-byte loads in flight per lane),
// summed in fp32 in copy order k = 0..K-1 (then the shared expert's row),
// and stored as bf16.
template <int NB>   // copies whose loads are issued together
__global__ void __launch_bounds__(256) combine_kernel(int n_tok, int d8, int K, const uint4* __restrict__ y_perm,
                                                      const int32_t* __restrict__ row_of_copy,
                                                      const float* __restrict__ topk_w,
                                                      const uint4* __restrict__ y_shared, uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int segs = (d8 + 127) / 128;
  const int64_t items = static_cast<int64_t>(n_tok) * segs;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
       it += wstride) {
    const int t = static_cast<int>(it / segs);
    const int i0 = static_cast<int>(it - static_cast<int64_t>(t) * segs) * 128 + lane;
    float acc[4][8];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) acc[qq][jj] = 0.0f;
    // a dropped copy (capacity mode) or a slot past K adds 0 * 0, which
    // leaves acc unchanged (acc, a sum started at +0, is never -0)
    for (int k0 = 0; k0 < K; k0 += NB) {
      uint4 v[NB][4];
      float wk[NB];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int k = k0 + j;
        const int r = k < K ? __ldg(row_of_copy + static_cast<int64_t>(t) * K + k) : -1;
        wk[j] = r >= 0 ? __ldg(topk_w + static_cast<int64_t>(t) * K + k) : 0.0f;
        const uint4* src = y_perm + static_cast<int64_t>(r >= 0 ? r : 0) * d8;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int i = i0 + 32 * qq;
          v[j][qq] = (r >= 0 && i < d8) ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          float y[8];
          unpack8(v[j][qq], y);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) acc[qq][jj] = fmaf(wk[j], y[jj], acc[qq][jj]);
        }
      }
    }
    if (y_shared) {
      uint4 sv[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int i = i0 + 32 * qq;
        sv[qq] = i < d8 ? __ldg(y_shared + static_cast<int64_t>(t) * d8 + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float y[8];
        unpack8(sv[qq], y);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[qq][jj] += y[jj];
      }
    }
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int i = i0 + 32 * qq;
      if (i < d8) out[static_cast<int64_t>(t) * d8 + i] = pack8(acc[qq]);
    }
  }
}

// ------------------------------------------------------------ combine backward
constexpr int kMaxK = 32;

template <int NB>
__global__ void __launch_bounds__(256, 3) combine_bwd_kernel(int n_tok, int d8, int K, int gate, int E,
                                                          const uint4* __restrict__ dy,
                                                          const uint4* __restrict__ y_perm,
                                                          const int32_t* __restrict__ row_of_copy,
                                                          const float* __restrict__ topk_w,
                                                          const float* __restrict__ logits,
                                                          const int32_t* __restrict__ topk_idx,
                                                          uint4* __restrict__ dyw, float* __restrict__ dg_out,
                                                          float* __restrict__ dl_out, uint8_t* __restrict__ q_codes,
                                                          uint8_t* __restrict__ q_scales, int64_t q_ld) {
  __shared__ int s_rows[kMaxK];
  __shared__ float s_w[kMaxK];
  __shared__ float s_part[8][kMaxK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < K) {
      s_rows[threadIdx.x] = row_of_copy[static_cast<int64_t>(t) * K + threadIdx.x];
      s_w[threadIdx.x] = topk_w[static_cast<int64_t>(t) * K + threadIdx.x];
    }
    __syncthreads();
    float part[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) part[k] = 0.0f;
    // A warp covers 32 consecutive 8-column chunks per pass and stays
    // converged (the pass count is uniform per warp), so with q_codes the
    // four lanes of each 32-column block combine their block maxima by
    // shuffles.
    for (int i0 = warp * 32; i0 < d8; i0 += blockDim.x) {
      const int i = i0 + lane;
      const bool act = i < d8;
      float g8[8];
      if (act) {
        unpack8(dy[static_cast<int64_t>(t) * d8 + i], g8);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) g8[j] = 0.0f;
      }
      // copies in groups of NB: their y_perm loads are issued together
#pragma unroll
      for (int k0 = 0; k0 < kMaxK; k0 += NB) {
        if (k0 >= K) break;
        uint4 u[NB];
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          const int rr = k0 + c < K ? s_rows[k0 + c] : -1;
          u[c] = (act && rr >= 0) ? y_perm[static_cast<int64_t>(rr) * d8 + i] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          const int k = k0 + c;
          if (k >= K || s_rows[k] < 0) continue;   // a dropped copy has no row and dg = 0
          const int64_t r = s_rows[k];
          float y[8], o[8];
          unpack8(u[c], y);
          const float w = s_w[k];
          float acc = 0.0f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc = fmaf(g8[j], y[j], acc);
            o[j] = w * g8[j];
          }
          part[k] += acc;
          const uint4 packed = pack8(o);
          if (act) dyw[r * d8 + i] = packed;
          if (q_codes) {
            // MXFP8 copy of the stored (bf16) dYw row along D
            float v[8];
            unpack8(packed, v);
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int e = mx_scale_exponent(amax);
            if (act) {
              *reinterpret_cast<uint2*>(q_codes + r * (8 * static_cast<int64_t>(d8)) + 8 * i) =
                  mx_encode8(v, mx_inv_scale(e));
              if ((i & 3) == 0) q_scales[static_cast<int64_t>(i >> 2) * q_ld + r] = static_cast<uint8_t>(e + 127);
            }
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      if (k < K) {
        const float v = warp_sum(part[k]);
        if (lane == 0) s_part[warp][k] = v;
      }
    }
    __syncthreads();
    if (warp == 0) {
      float dgk = 0.0f, gk = 0.0f, lk = 0.0f;
      if (lane < K) {
        for (int w = 0; w < 8; ++w) dgk += s_part[w][lane];
        gk = s_w[lane];
        if (gate == 1) lk = logits[static_cast<int64_t>(t) * E + topk_idx[static_cast<int64_t>(t) * K + lane]];
      }
      const float inner = warp_sum(lane < K ? gk * dgk : 0.0f);
      float dl = 0.0f;
      if (gate == 0) {
        dl = gk * (dgk - inner);
      } else {
        const float sg = (lane < K) ? 1.0f / (1.0f + expf(-lk)) : 0.0f;
        const float ssum = warp_sum(sg);
        dl = (lane < K) ? sg * (1.0f - sg) / ssum * (dgk - inner) : 0.0f;
      }
      if (lane < K) {
        if (dg_out) dg_out[static_cast<int64_t>(t) * K + lane] = dgk;
        dl_out[static_cast<int64_t>(t) * K + lane] = dl;
      }
    }
  }
}

// ------------------------------------------------------------ router weight gradient
// dW_g[e] = sum over the rows r of expert e of dl[copy_of_row[r]] * x_perm[r].
// Ragged and deterministic: every expert's rows are cut into 64-row chunks
// (chunk list derived on the device from the offsets), each chunk's partial
// sum is written once, and the partials of an expert are added in chunk order.
constexpr int kDwgChunk = 64;

__global__ void dwg_chunk_prefix_kernel(int E, const int32_t* __restrict__ offsets, int32_t* __restrict__ cpre) {
  // single warp: prefix of ceil(m_e / 64) over the experts
  const int lane = threadIdx.x;
  const int per = (E + 31) / 32;
  const int lo = lane * per, hi = min(E, lo + per);
  int sum = 0;
  for (int e = lo; e < hi; ++e) sum += max(0, offsets[e + 1] - offsets[e] + kDwgChunk - 1) / kDwgChunk;
  int incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  int run = incl - sum;
  for (int e = lo; e < hi; ++e) {
    cpre[e] = run;
    run += max(0, offsets[e + 1] - offsets[e] + kDwgChunk - 1) / kDwgChunk;
  }
  if (lane == 31) cpre[E] = incl;
}

__global__ void __launch_bounds__(256) dwg_partial_kernel(int E, int d8, const int32_t* __restrict__ offsets,
                                                          const int32_t* __restrict__ cpre,
                                                          const int32_t* __restrict__ copy_of_row,
                                                          const float* __restrict__ dl,
                                                          const uint4* __restrict__ x_rows, int gather_k,
                                                          float* __restrict__ partial) {
  __shared__ float s_w[kDwgChunk];
  __shared__ int s_row[kDwgChunk];
  __shared__ int s_e;
  const int c = blockIdx.x;
  if (c >= cpre[E]) return;                      // uniform across the block
  if (threadIdx.x == 0) {
    int lo = 0, hi = E;                          // largest e with cpre[e] <= c
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cpre[mid] <= c) lo = mid; else hi = mid;
    }
    s_e = lo;
  }
  __syncthreads();
  const int e = s_e;
  const int r0 = offsets[e] + (c - cpre[e]) * kDwgChunk;
  const int n = min(kDwgChunk, offsets[e + 1] - r0);
  if (threadIdx.x < n) {
    // permuted row r0 + t: a row of x_perm, or (gather_k > 0) token row copy / K of x
    const int cp = copy_of_row[r0 + threadIdx.x];
    s_w[threadIdx.x] = dl[cp];
    s_row[threadIdx.x] = gather_k > 0 ? cp / gather_k : r0 + threadIdx.x;
  }
  __syncthreads();
  const int i = blockIdx.y * blockDim.x + threadIdx.x;
  if (i >= d8) return;
  const uint4* src = x_rows + i;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int j = 0;
  for (; j + 4 <= n; j += 4) {
    const uint4 v0 = src[static_cast<int64_t>(s_row[j]) * d8];
    const uint4 v1 = src[static_cast<int64_t>(s_row[j + 1]) * d8];
    const uint4 v2 = src[static_cast<int64_t>(s_row[j + 2]) * d8];
    const uint4 v3 = src[static_cast<int64_t>(s_row[j + 3]) * d8];
    float x0[8], x1[8], x2[8], x3[8];
    unpack8(v0, x0);
    unpack8(v1, x1);
    unpack8(v2, x2);
    unpack8(v3, x3);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      acc[q] = fmaf(s_w[j], x0[q], acc[q]);
      acc[q] = fmaf(s_w[j + 1], x1[q], acc[q]);
      acc[q] = fmaf(s_w[j + 2], x2[q], acc[q]);
      acc[q] = fmaf(s_w[j + 3], x3[q], acc[q]);
    }
  }
  for (; j < n; ++j) {
    float x[8];
    unpack8(src[static_cast<int64_t>(s_row[j]) * d8], x);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = fmaf(s_w[j], x[q], acc[q]);
  }
  float4* dst = reinterpret_cast<float4*>(partial + static_cast<int64_t>(c) * d8 * 8) + 2 * i;
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__global__ void __launch_bounds__(256) dwg_reduce_kernel(int E, int d, const int32_t* __restrict__ cpre,
                                                         const float* __restrict__ partial, float* __restrict__ out) {
  const int e = blockIdx.x;
  const int i = blockIdx.y * blockDim.x + threadIdx.x;
  if (i * 4 >= d) return;
  const int c0 = cpre[e], c1 = cpre[e + 1];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = c0; c < c1; ++c) {
    const float4 v = reinterpret_cast<const float4*>(partial + static_cast<int64_t>(c) * d)[i];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  reinterpret_cast<float4*>(out + static_cast<int64_t>(e) * d)[i] = acc;
}

// ------------------------------------------------------------ unpermute-sum of dx
template <int NB>
__global__ void __launch_bounds__(256) unpermute_dx_kernel(int n_tok, int d8, int K, const uint4* __restrict__ dx_perm,
                                                           const int32_t* __restrict__ row_of_copy,
                                                           const float* __restrict__ dl,
                                                           const int32_t* __restrict__ topk_idx,
                                                           const uint4* __restrict__ w_gate,
                                                           const uint4* __restrict__ dx_shared,
                                                           uint4* __restrict__ dx) {
  __shared__ int s_rows[32];
  __shared__ int s_e[32];
  __shared__ float s_dl[32];
  for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < K) {
      const int64_t c = static_cast<int64_t>(t) * K + threadIdx.x;
      s_rows[threadIdx.x] = row_of_copy[c];
      s_e[threadIdx.x] = topk_idx[c];
      s_dl[threadIdx.x] = dl ? dl[c] : 0.0f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < d8; i += blockDim.x) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      // NB copies' loads in flight at once; a dropped copy (no expert
      // gradient) or a slot past K adds +0, which leaves acc unchanged (acc,
      // a sum started at +0, is never -0)
      for (int k0 = 0; k0 < K; k0 += NB) {
        uint4 u[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const int r = k0 + j < K ? s_rows[k0 + j] : -1;
          u[j] = r >= 0 ? dx_perm[static_cast<int64_t>(r) * d8 + i] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          float v[8];
          unpack8(u[j], v);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) acc[jj] += v[jj];
        }
      }
      if (w_gate && dl) {
        for (int k0 = 0; k0 < K; k0 += NB) {
          uint4 u[NB];
          float wk[NB];
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            const bool in = k0 + j < K;
            u[j] = in ? w_gate[static_cast<int64_t>(s_e[k0 + j]) * d8 + i] : make_uint4(0, 0, 0, 0);
            wk[j] = in ? s_dl[k0 + j] : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            float v[8];
            unpack8(u[j], v);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) acc[jj] = fmaf(wk[j], v[jj], acc[jj]);
          }
        }
      }
      if (dx_shared) {
        float v[8];
        unpack8(dx_shared[static_cast<int64_t>(t) * d8 + i], v);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += v[j];
      }
      dx[static_cast<int64_t>(t) * d8 + i] = pack8(acc);
    }
  }
}

// ------------------------------------------------------------ capacity (drop) mode
// Kept copies per expert min(count, cap), their exclusive scan, and the
// number of dropped copies (single block, E <= 1024).
__global__ void __launch_bounds__(1024) kept_offsets_kernel(const int32_t* __restrict__ offsets, int E, int cap,
                                                            int total, int32_t* __restrict__ kept_offsets,
                                                            int32_t* __restrict__ n_dropped) {
  __shared__ int32_t s[1024];
  const int e = threadIdx.x;
  const int32_t v = e < E ? min(offsets[e + 1] - offsets[e], cap) : 0;
  s[e] = v;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    const int32_t add = e >= d ? s[e - d] : 0;
    __syncthreads();
    s[e] += add;
    __syncthreads();
  }
  if (e < E) kept_offsets[e + 1] = s[e];
  if (e == 0) {
    kept_offsets[0] = 0;
    if (n_dropped) *n_dropped = total - s[1023];
  }
}

// Copy c keeps its rank inside its expert (position in the dropless,
// token-ordered permutation); ranks below the capacity get the compact row
// kept_offsets[e] + rank, the others -1.
// A copy without a dropless row (expert index outside [0, E), or offsets
// inconsistent with the indices, both reported by the map kernels) is dropped.
__global__ void capacity_rows_kernel(int64_t R, int E, const int32_t* __restrict__ idx,
                                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_full,
                                     const int32_t* __restrict__ kept_offsets, int cap,
                                     int32_t* __restrict__ row_of_copy, int32_t* __restrict__ copy_of_row) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= R) return;
  const int e = idx[c];
  const int rf = row_full[c];
  int32_t r = -1;
  const int rank = (e >= 0 && e < E && rf >= 0) ? rf - offsets[e] : cap;
  if (rank >= 0 && rank < cap) {
    r = kept_offsets[e] + rank;
    copy_of_row[r] = static_cast<int32_t>(c);
  }
  row_of_copy[c] = r;
}

__global__ void dense_offsets_kernel(int32_t* dst, int n) {
  if (threadIdx.x == 0) {
    dst[0] = 0;
    dst[1] = n;
  }
}

int num_sms_kernels() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 128;
}

int grid_for_tokens(int n_tok) {
  const int g = num_sms_kernels() * 8;
  return n_tok < g ? (n_tok > 0 ? n_tok : 1) : g;
}

}  // namespace

cudaError_t launch_topk_scan(const RouteShape& s, const float* part, int ks, float* logits, const float* bias,
                             int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* acc,
                             int32_t* ticket, int32_t* status, cudaStream_t st) {
  if (s.n_tok <= 0) return cudaSuccess;
  if (s.n_exp > 1024 || ks < 1 || ks > kTopkMaxSlices) return cudaErrorInvalidValue;
  const int blocks = (s.n_tok + 7) / 8;
  const size_t smem = static_cast<size_t>(s.n_exp) * sizeof(int);
  const int pl = (s.n_exp + 31) / 32;
#define MOE_TOPK_SCAN(P)                                                                                          \
  topk_scan_kernel<P><<<blocks, 256, smem, st>>>(s, part, ks, logits, bias, topk_idx, topk_w, counts, offsets, acc, \
                                                 ticket, status)
  if (pl <= 1) MOE_TOPK_SCAN(1);
  else if (pl <= 2) MOE_TOPK_SCAN(2);
  else if (pl <= 4) MOE_TOPK_SCAN(4);
  else if (pl <= 8) MOE_TOPK_SCAN(8);
  else if (pl <= 16) MOE_TOPK_SCAN(16);
  else MOE_TOPK_SCAN(32);
#undef MOE_TOPK_SCAN
  return cudaGetLastError();
}

cudaError_t launch_router_fused(const RouteShape& s, int d, const void* x, const void* w_gate, const float* bias,
                                float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                int32_t* acc, int32_t* ticket, int32_t* status, cudaStream_t st) {
  if (s.n_tok <= 0 || s.n_exp > 32 || d % 32) return cudaErrorInvalidValue;
  const int blocks = static_cast<int>((static_cast<int64_t>(s.n_tok) + kRtTok - 1) / kRtTok);
  const int nt = (s.n_exp + 7) / 8;
#define MOE_ROUTER(NT)                                                                                            \
  router_fused_kernel<NT><<<blocks, kRtWarps * 32, 0, st>>>(s, d / 8, static_cast<const uint4*>(x),               \
                                                            static_cast<const uint4*>(w_gate), bias, logits,       \
                                                            topk_idx, topk_w, counts, offsets, acc, ticket, status)
  if (nt <= 1) MOE_ROUTER(1);
  else if (nt <= 2) MOE_ROUTER(2);
  else MOE_ROUTER(4);
#undef MOE_ROUTER
  return cudaGetLastError();
}

// At most this many CTAs of route_permute_kernel are resident at once (two
// per SM by its launch bounds): the tile count may exceed ceil(N/16) by that.
constexpr int kRpMaxGrid = 2048;

int64_t route_permute_hist_words(int n_tok, int n_exp) {
  // arrivals and generation words (two 128-byte lines), then T x E histograms
  return 64 + ((static_cast<int64_t>(n_tok) + kRtTok - 1) / kRtTok + kRpMaxGrid) * n_exp;
}

cudaError_t launch_route_permute(const RouteShape& s, int d, const void* x, const void* w_gate, const float* bias,
                                 float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                 int32_t* row_of_copy, int32_t* copy_of_row, void* x_perm, int32_t* ws_words,
                                 int32_t* status, cudaStream_t st) {
  if (s.n_tok <= 0 || s.n_exp > 32 || s.top_k > 32 || d % 32) return cudaErrorInvalidValue;
  const int t16 = static_cast<int>((static_cast<int64_t>(s.n_tok) + kRtTok - 1) / kRtTok);
  const int nt = (s.n_exp + 7) / 8;
  auto go = [&](auto kern) -> cudaError_t {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRtWarps * 32, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int g = std::min(per_sm * num_sms_kernels(), kRpMaxGrid);
    // tiles: ceil(N/16) when that is under half the grid (a small batch);
    // otherwise rounded up to a multiple of the grid, so every CTA routes and
    // copies the same number of tiles
    const int ntiles = t16 * 2 < g ? t16 : (t16 + g - 1) / g * g;
    const int blocks = std::min(ntiles, g);
    RouteShape sa = s;
    int d8 = d / 8;
    int nti = ntiles, tq = s.n_tok / ntiles, trem = s.n_tok % ntiles;
    const uint4* xa = static_cast<const uint4*>(x);
    const uint4* wa = static_cast<const uint4*>(w_gate);
    uint4* xp = static_cast<uint4*>(x_perm);
    int32_t* bar = ws_words;
    int32_t* th = ws_words + 64;
    void* args[] = {&sa, &d8, &nti, &tq, &trem, &xa, &wa, const_cast<float**>(&bias), &logits, &topk_idx, &topk_w, &counts,
                    &offsets, &row_of_copy, &copy_of_row, &xp, &th, &bar, &status};
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kRtWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kern), args);
  };
  if (nt <= 1) return go(route_permute_kernel<1>);
  if (nt <= 2) return go(route_permute_kernel<2>);
  return go(route_permute_kernel<4>);
}

cudaError_t launch_update_bias(const int32_t* counts, int n_exp, float* bias, float gamma, int mode,
                               cudaStream_t st) {
  const float target = static_cast<float>(1.0 / static_cast<double>(n_exp));
  update_bias_kernel<<<1, 256, 0, st>>>(counts, n_exp, bias, gamma, mode, target);
  return cudaGetLastError();
}

int permute_num_chunks(int n_tok) { return (n_tok + kChunkTok - 1) / kChunkTok; }

cudaError_t launch_permute_maps(int n_tok, int n_exp, int top_k, const int32_t* topk_idx, const int32_t* offsets,
                                int32_t* block_counts, int32_t* block_base, int32_t* row_of_copy,
                                int32_t* copy_of_row, int32_t* status, cudaStream_t st, bool chunked) {
  if (n_tok <= 0) return cudaSuccess;
  if (!chunked && static_cast<int64_t>(n_tok) * top_k <= kMapOnePassMax) {
    const size_t smem = static_cast<size_t>(33) * n_exp * sizeof(int);
    if (smem > 48 * 1024) {   // above the default dynamic shared-memory limit (more than 372 experts)
      const cudaError_t e = cudaFuncSetAttribute(maps_onepass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    maps_onepass_kernel<<<1, 1024, smem, st>>>(n_tok, n_exp, top_k, topk_idx, offsets, row_of_copy, copy_of_row,
                                               status);
    return cudaGetLastError();
  }
  const int nch = permute_num_chunks(n_tok);
  const size_t smem = static_cast<size_t>(n_exp) * sizeof(int);
  block_hist_kernel<<<nch, 256, smem, st>>>(n_tok, n_exp, top_k, topk_idx, block_counts, status);
  block_base_kernel<<<(n_exp + 255) / 256, 256, 0, st>>>(nch, n_exp, offsets, block_counts, block_base, status);
  scatter_maps_kernel<<<nch, 32, 2 * smem, st>>>(n_tok, n_exp, top_k, topk_idx, offsets, block_base, row_of_copy,
                                                 copy_of_row, status);
  return cudaGetLastError();
}

int64_t permute_single_pass_look_words(int n_tok, int n_exp) {
  return (static_cast<int64_t>(n_tok) + kSpTok - 1) / kSpTok * n_exp;
}

cudaError_t launch_permute_single_pass(int n_tok, int n_exp, int top_k, int d, const int32_t* topk_idx,
                                       const int32_t* offsets, const void* x, int32_t* row_of_copy,
                                       int32_t* copy_of_row, void* x_perm, unsigned long long* look, int32_t* ctl,
                                       int32_t* status, cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  if (top_k > 32 || d % 8) return cudaErrorInvalidValue;
  const int chunks = (n_tok + kSpTok - 1) / kSpTok;
  const size_t smem = (2 * static_cast<size_t>(n_exp) + 2 * kSpTok * top_k) * sizeof(int);
  permute_single_pass_kernel<false><<<chunks, kSpThreads, smem, st>>>(
      n_tok, n_exp, top_k, d / 8, topk_idx, offsets, static_cast<const uint4*>(x), row_of_copy, copy_of_row,
      static_cast<uint4*>(x_perm), look, ctl, status, SpQuantOut{});
  return cudaGetLastError();
}

cudaError_t launch_permute_single_pass_mxfp8(int n_tok, int n_exp, int top_k, int d, const int32_t* topk_idx,
                                             const int32_t* offsets, const void* x, int32_t* row_of_copy,
                                             int32_t* copy_of_row, uint8_t* codes, uint8_t* scales, int64_t ld,
                                             uint8_t* tok_codes, uint8_t* tok_scales, int64_t tok_ld,
                                             unsigned long long* look, int32_t* ctl, int32_t* status,
                                             cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  if (top_k > 32 || d % 32) return cudaErrorInvalidValue;
  const int chunks = (n_tok + kSpTok - 1) / kSpTok;
  const size_t smem = (2 * static_cast<size_t>(n_exp) + 2 * kSpTok * top_k) * sizeof(int);
  permute_single_pass_kernel<true><<<chunks, kSpThreads, smem, st>>>(
      n_tok, n_exp, top_k, d / 8, topk_idx, offsets, static_cast<const uint4*>(x), row_of_copy, copy_of_row,
      nullptr, look, ctl, status, SpQuantOut{codes, scales, ld, tok_codes, tok_scales, tok_ld});
  return cudaGetLastError();
}

cudaError_t launch_permute_rows(int n_tok, int d, int top_k, const void* x, const int32_t* row_of_copy,
                                void* x_perm, cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  permute_rows_kernel<<<grid_for_tokens(n_tok), 256, 0, st>>>(n_tok, d / 8, top_k, static_cast<const uint4*>(x),
                                                              row_of_copy, static_cast<uint4*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_combine(int n_tok, int d, int top_k, const void* y_perm, const int32_t* row_of_copy,
                           const float* topk_w, const void* y_shared, void* out, cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  auto kern = top_k == 1 ? combine_kernel<1> : (top_k == 2 ? combine_kernel<2> : combine_kernel<4>);
  const int64_t items = static_cast<int64_t>(n_tok) * ((d / 8 + 127) / 128);   // one warp each
  const int blocks = static_cast<int>(std::min<int64_t>((items + 7) / 8, static_cast<int64_t>(num_sms_kernels()) * 8));
  kern<<<blocks, 256, 0, st>>>(n_tok, d / 8, top_k, static_cast<const uint4*>(y_perm), row_of_copy, topk_w,
                               static_cast<const uint4*>(y_shared), static_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(int n_tok, int d, int top_k, int gate, const void* dy, const void* y_perm,
                               const int32_t* row_of_copy, const float* topk_w, const float* logits, int n_exp,
                               const int32_t* topk_idx, void* dyw, float* dg, float* dl, cudaStream_t st,
                               uint8_t* q_codes, uint8_t* q_scales, int64_t q_ld) {
  if (n_tok <= 0) return cudaSuccess;
  if (top_k > kMaxK || (q_codes && (d % 32 != 0 || !q_scales))) return cudaErrorInvalidValue;
  auto kern = top_k == 1 ? combine_bwd_kernel<1> : (top_k == 2 ? combine_bwd_kernel<2> : combine_bwd_kernel<4>);
  kern<<<grid_for_tokens(n_tok), 256, 0, st>>>(
      n_tok, d / 8, top_k, gate, n_exp, static_cast<const uint4*>(dy), static_cast<const uint4*>(y_perm),
      row_of_copy, topk_w, logits, topk_idx, static_cast<uint4*>(dyw), dg, dl, q_codes, q_scales, q_ld);
  return cudaGetLastError();
}

size_t dwgate_partial_floats(int n_tok, int top_k, int n_exp, int d) {
  const size_t chunks = (static_cast<size_t>(n_tok) * top_k + kDwgChunk - 1) / kDwgChunk + n_exp;
  return chunks * d + (n_exp + 1 + 3) / 4 * 4;   // partials + chunk prefix (int32)
}

cudaError_t launch_dwgate(int n_tok, int top_k, int n_exp, int d, const int32_t* offsets, const int32_t* copy_of_row,
                          const float* dl, const void* x_rows, int gather_k, float* scratch, float* dw_gate,
                          cudaStream_t st) {
  if (n_exp > 1024 || !scratch) return cudaErrorInvalidValue;
  const int chunks = static_cast<int>((static_cast<int64_t>(n_tok) * top_k + kDwgChunk - 1) / kDwgChunk + n_exp);
  float* partial = scratch;
  int32_t* cpre = reinterpret_cast<int32_t*>(scratch + static_cast<size_t>(chunks) * d);
  const int d8 = d / 8;
  dwg_chunk_prefix_kernel<<<1, 32, 0, st>>>(n_exp, offsets, cpre);
  dwg_partial_kernel<<<dim3(chunks, (d8 + 255) / 256), 256, 0, st>>>(
      n_exp, d8, offsets, cpre, copy_of_row, dl, static_cast<const uint4*>(x_rows), gather_k, partial);
  dwg_reduce_kernel<<<dim3(n_exp, (d / 4 + 255) / 256), 256, 0, st>>>(n_exp, d, cpre, partial, dw_gate);
  return cudaGetLastError();
}

cudaError_t launch_unpermute_dx(int n_tok, int d, int top_k, const void* dx_perm, const int32_t* row_of_copy,
                                const float* dl, const int32_t* topk_idx, const void* w_gate,
                                const void* dx_shared, void* dx, cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  auto kern = top_k == 1 ? unpermute_dx_kernel<1> : (top_k == 2 ? unpermute_dx_kernel<2> : unpermute_dx_kernel<4>);
  kern<<<grid_for_tokens(n_tok), 256, 0, st>>>(
      n_tok, d / 8, top_k, static_cast<const uint4*>(dx_perm), row_of_copy, dl, topk_idx,
      static_cast<const uint4*>(w_gate), static_cast<const uint4*>(dx_shared), static_cast<uint4*>(dx));
  return cudaGetLastError();
}

cudaError_t launch_capacity_maps(int n_tok, int n_exp, int top_k, const int32_t* topk_idx, const int32_t* offsets,
                                 const int32_t* row_full, int cap, int32_t* kept_offsets, int32_t* row_of_copy,
                                 int32_t* copy_of_row, int32_t* n_dropped, cudaStream_t st) {
  if (n_exp > 1024 || cap < 0) return cudaErrorInvalidValue;
  const int64_t R = static_cast<int64_t>(n_tok) * top_k;
  kept_offsets_kernel<<<1, 1024, 0, st>>>(offsets, n_exp, cap, static_cast<int>(R), kept_offsets, n_dropped);
  if (R > 0)
    capacity_rows_kernel<<<static_cast<unsigned>((R + 255) / 256), 256, 0, st>>>(R, n_exp, topk_idx, offsets, row_full,
                                                                                   kept_offsets, cap, row_of_copy,
                                                                                   copy_of_row);
  return cudaGetLastError();
}

cudaError_t launch_dense_offsets(int32_t* dst, int n, cudaStream_t st) {
  dense_offsets_kernel<<<1, 32, 0, st>>>(dst, n);
  return cudaGetLastError();
}

}  // namespace moe
