// C ABI of libmoe (declared in include/moe.h): argument validation,
// workspace layout, and the launch sequence of each entry point.
#include "moe.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "balance.cuh"
#include "grouped_gemm.cuh"
#include "moe_kernels.cuh"
#include "mxfp8.cuh"
#include "timing.cuh"

#include <nvtx3/nvToolsExt.h>

namespace {

using moe::GemmArgs;
using moe::Operand;

constexpr size_t kAlign = 256;
// int32 words of the workspace's status block (256 bytes, cleared by
// moe_workspace_init): 0 and 1 are the status bits and the failing site;
// the fused router keeps its completion ticket in word 8 and its histogram
// accumulator in words 16..47, and leaves both zero;
constexpr int kTicketWord = 8;
constexpr int kRouterAccWord = 16;
// words 48..50: the single-pass permute's chunk ticket, done counter and
// generation (it leaves the first two zero and advances the third)
constexpr int kPermuteCtlWord = 48;
// Look-back words of the single-pass permute (1 MiB): ceil(N/16) * E of them
// per call; larger problems take the two-kernel permute.
constexpr size_t kLookWords = 131072;
// The router tail's expert histogram accumulator (one int32 per expert, up to
// 1024), a fixed region like the look-back words; the kernel leaves it zero.
constexpr size_t kRouteAccWords = 1024;
// The router logits GEMM has one 128-token tile per CTA; with few tiles its
// contraction is cut into up to this many slices (summed in order after).
constexpr int kGateSlices = 4;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  size_t status = 0, dense_off = 0, blk_counts = 0, blk_base = 0, look = 0, racc = 0, aux = 0, gpart = 0,
         rp_hist = 0, fwd_end = 0;
  size_t hq = 0, hs = 0, hq_sh = 0, hs_sh = 0;   // MXFP8 h between GEMM1 and GEMM2
  size_t dl = 0, dg = 0, dyw = 0, da1 = 0, da3 = 0, da1s = 0, da3s = 0, dxs = 0, dwg = 0, gmaps = 0, total = 0;
  // MXFP8 backward: row-wise codes/scales of dYw, da1, da3 (dgrad operands),
  // padded group starts, and four transposed token-blocked code matrices
  // (weight-gradient operands: two [D, Rp], two [max(F,Fs), Rp]) with scales
  size_t q_dy = 0, q_dys = 0, q_da1 = 0, q_da1s = 0, q_da3 = 0, q_da3s = 0, pad = 0, pad_sh = 0;
  size_t t_d0 = 0, t_d0s = 0, t_d1 = 0, t_d1s = 0, t_f0 = 0, t_f0s = 0, t_f1 = 0, t_f1s = 0;
  int64_t rp = 0;   // leading dimension of the transposed code matrices
};

int64_t ld16(int64_t v) { return (v + 15) / 16 * 16; }

WsLayout layout(const moe_desc_t& d) {
  WsLayout L;
  const size_t N = d.n_tok, D = d.d_model, F = d.d_ff, E = d.n_exp, K = d.top_k;
  const size_t R = N * K, Fs = d.n_shared ? d.d_ff_shared : 0;
  const size_t nch = moe::permute_num_chunks(d.n_tok);
  size_t o = 0;
  L.status = o; o += kAlign;
  L.dense_off = o; o += kAlign;
  // the single-pass permute's look-back words: a fixed region of the same
  // place and size for every description, holding nothing else
  L.look = o; o += kLookWords * 8;
  L.racc = o; o += kRouteAccWords * 4;
  L.blk_counts = o; o = align_up(o + nch * E * 4);
  L.blk_base = o; o = align_up(o + nch * E * 4);
  L.aux = o; o = align_up(o + moe::aux_partial_floats(d.n_tok > 0 ? d.n_tok : 1, d.n_exp) * 4);
  L.gpart = o; o = align_up(o + static_cast<size_t>(kGateSlices) * N * E * 4);   // router logit slices
  // moe_route_permute's grid-barrier words and per-tile expert histograms (E <= 32)
  L.rp_hist = o;
  o = align_up(o + (E <= 32 ? static_cast<size_t>(moe::route_permute_hist_words(d.n_tok, d.n_exp)) * 4 + 128 : 0));
  if (d.precision == 1) {
    L.hq = o; o = align_up(o + R * F);
    L.hs = o; o = align_up(o + F / 32 * moe::mx_scale_ld(R));
    L.hq_sh = o; o = align_up(o + N * Fs);
    L.hs_sh = o; o = align_up(o + Fs / 32 * moe::mx_scale_ld(N));
  }
  L.fwd_end = o;
  L.dl = o; o = align_up(o + R * 4);
  L.dg = o; o = align_up(o + R * 4);
  L.dyw = o; o = align_up(o + R * D * 2);  // also holds dx_perm
  L.da1 = o; o = align_up(o + R * F * 2);
  L.da3 = o; o = align_up(o + R * F * 2);
  L.da1s = o; o = align_up(o + N * Fs * 2);
  L.da3s = o; o = align_up(o + N * Fs * 2);
  L.dxs = o; o = align_up(o + (Fs ? N * D * 2 : 0));
  L.dwg = o; o = align_up(o + moe::dwgate_partial_floats(d.n_tok, d.top_k, d.n_exp, d.d_model) * 4);
  // per-group maps of the weight gradients (+128 bytes: the workspace itself
  // is only 16-byte aligned, the maps need 128)
  L.gmaps = o; o = align_up(o + moe::kGemmMapScratchBytes + 128);
  if (d.precision == 1) {
    const size_t Fm = F > Fs ? F : Fs;
    const size_t ldr = moe::mx_scale_ld(R);
    L.q_dy = o; o = align_up(o + R * D);
    L.q_dys = o; o = align_up(o + D / 32 * ldr);
    L.q_da1 = o; o = align_up(o + R * Fm);
    L.q_da1s = o; o = align_up(o + Fm / 32 * ldr);
    L.q_da3 = o; o = align_up(o + R * Fm);
    L.q_da3s = o; o = align_up(o + Fm / 32 * ldr);
    L.pad = o; o = align_up(o + (E + 1) * 4);
    L.pad_sh = o; o = align_up(o + 2 * 4);
    L.rp = (moe::mx_padded_rows(static_cast<int64_t>(R), static_cast<int>(E)) + 127) / 128 * 128;
    const size_t rp = static_cast<size_t>(L.rp);
    L.t_d0 = o; o = align_up(o + D * rp);
    L.t_d0s = o; o = align_up(o + rp / 32 * ld16(D));
    L.t_d1 = o; o = align_up(o + D * rp);
    L.t_d1s = o; o = align_up(o + rp / 32 * ld16(D));
    L.t_f0 = o; o = align_up(o + Fm * rp);
    L.t_f0s = o; o = align_up(o + rp / 32 * ld16(Fm));
    L.t_f1 = o; o = align_up(o + Fm * rp);
    L.t_f1s = o; o = align_up(o + rp / 32 * ld16(Fm));
  }
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}
// The 128-byte-aligned start of the weight gradients' map scratch.
void* map_scratch(void* ws, const WsLayout& L) {
  const uintptr_t p = reinterpret_cast<uintptr_t>(static_cast<char*>(ws) + L.gmaps);
  return reinterpret_cast<void*>((p + 127) & ~uintptr_t(127));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_desc(const moe_desc_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->n_tok < 0 || d->d_model <= 0 || d->d_ff <= 0 || d->n_exp <= 0 || d->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (d->top_k > d->n_exp || d->top_k > 32 || d->n_exp > 1024) return MOE_ERR_INVALID_ARG;
  if (d->d_model % 64 || d->d_ff % 64) return MOE_ERR_INVALID_ARG;
  if (d->gate != 0 && d->gate != 1) return MOE_ERR_INVALID_ARG;
  if (d->use_bias != 0 && d->use_bias != 1) return MOE_ERR_INVALID_ARG;
  if (d->n_shared != 0 && d->n_shared != 1) return d->n_shared > 1 ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
  if (d->n_shared && (d->d_ff_shared <= 0 || d->d_ff_shared % 64)) return MOE_ERR_INVALID_ARG;
  if (d->precision < 0 || d->precision > 2) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->n_tok) * d->top_k >= (int64_t{1} << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_ws(const moe_desc_t& d, void* ws, size_t ws_bytes, bool bwd) {
  if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  const WsLayout L = layout(d);
  if (ws_bytes < (bwd ? L.total : L.fwd_end)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                          \
  do {                                         \
    const moe_status_t s_ = (expr);            \
    if (s_ != MOE_OK) return s_;               \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// Grouped-GEMM launch, timed under its kind while moe_timing is enabled.
cudaError_t gemm(int kind, const GemmArgs& a, cudaStream_t st) {
  return moe::timed(kind, st, [&] { return moe::launch_grouped_gemm(a, st); });
}

// NVTX range around an entry point's enqueue work (a no-op unless a
// profiler or tracer is attached to the process).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define MOE_RANGE(name) const NvtxRange moe_nvtx_range_(name)

bool all16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p || !aligned16(p)) return false;
  return true;
}

// A K-major activation [rows, cols] (row-major, ld = cols).
Operand act(const void* p, int64_t rows, int64_t cols) {
  Operand o;
  o.ptr = p;
  o.rows = rows;
  o.cols = cols;
  o.ld = cols;
  o.groups = 1;
  o.group_stride = rows * cols;
  return o;
}
// A stack of `groups` weight matrices [rows, cols] each.
Operand wstack(const void* p, int64_t groups, int64_t rows, int64_t cols) {
  Operand o = act(p, rows, cols);
  o.groups = groups;
  o.group_stride = rows * cols;
  return o;
}

// SwiGLU FFN of one "expert set": GEMM1 (fused w1|w3 with SwiGLU epilogue)
// then GEMM2, over `groups` ragged row groups of `a_in` [rows, D].
// (w8: w1, w3, w2 are E4M3 codes with fp32 tile scales s1, s3, s2)
// (gather: GEMM1's row r is row gather[r] / gather_k of a_in [n_src, D], read
// by TMA gathers instead of a permuted copy)
moe_status_t ffn_pair(const void* a_in, int64_t rows, int D, int F, int groups, const int32_t* offsets,
                      const void* w1, const void* w3, const void* w2, void* h, void* a1, void* a3, void* y,
                      int32_t* status, cudaStream_t st, const float* s1 = nullptr, const float* s3 = nullptr,
                      const float* s2 = nullptr, const int32_t* gather = nullptr, int gather_k = 0,
                      int64_t n_src = 0) {
  const bool w8 = s1 != nullptr;
  GemmArgs g1;
  g1.w8 = w8;
  g1.w8_scale[0] = s1;
  g1.w8_scale[1] = s3;
  g1.epi = moe::EPI_SWIGLU_FWD;
  g1.a[0] = act(a_in, gather ? n_src : rows, D);
  g1.a_gather = gather;
  g1.gather_k = gather_k;
  g1.b[0] = wstack(w1, groups, F, D);
  g1.b[1] = wstack(w3, groups, F, D);
  g1.b_dual_n = true;
  g1.k0 = D;
  g1.offsets = offsets;
  g1.num_groups = groups;
  g1.max_rows = rows;
  g1.n_size = F;
  g1.out0 = h;
  g1.out1 = a1;
  g1.out2 = a3;
  g1.ld_out = F;
  g1.status = status;
  MOE_CUDA(gemm(moe::TIMING_FFN_FWD, g1, st));
  GemmArgs g2;
  g2.w8 = w8;
  g2.w8_scale[0] = s2;
  g2.epi = moe::EPI_BF16;
  g2.a[0] = act(h, rows, F);
  g2.b[0] = wstack(w2, groups, D, F);
  g2.k0 = F;
  g2.offsets = offsets;
  g2.num_groups = groups;
  g2.max_rows = rows;
  g2.n_size = D;
  g2.out0 = y;
  g2.ld_out = D;
  g2.status = status;
  MOE_CUDA(gemm(moe::TIMING_FFN_FWD, g2, st));
  return MOE_OK;
}

// Backward of one expert set: dgrad through w2 with the SwiGLU derivative,
// weight gradient of w2, dgrad through w1|w3, weight gradients of w1, w3.
moe_status_t ffn_pair_bwd(const void* dyw, const void* a_in, const void* a1, const void* a3, const void* h,
                          int64_t rows, int D, int F, int groups, const int32_t* offsets, const void* w1,
                          const void* w3, const void* w2, void* da1, void* da3, void* dx_rows, float* dw1,
                          float* dw3, float* dw2, int32_t* status, cudaStream_t st, void* map_ws,
                          const float* s1 = nullptr, const float* s3 = nullptr, const float* s2 = nullptr) {
  const bool w8 = s1 != nullptr;   // FP8 weights in the data gradients; weight gradients stay bf16
  GemmArgs g;
  g.w8 = w8;
  g.w8_scale[0] = s2;
  g.epi = moe::EPI_SWIGLU_BWD;
  g.b_mn = true;
  g.a[0] = act(dyw, rows, D);
  g.b[0] = wstack(w2, groups, D, F);  // B[n=f, k=d], f contiguous
  g.k0 = D;
  g.offsets = offsets;
  g.num_groups = groups;
  g.max_rows = rows;
  g.n_size = F;
  g.in0 = a1;
  g.in1 = a3;
  g.out0 = da1;
  g.out1 = da3;
  g.ld_out = F;
  g.status = status;
  MOE_CUDA(gemm(moe::TIMING_DGRAD, g, st));

  GemmArgs w;
  w.epi = moe::EPI_F32;
  w.a_mn = w.b_mn = w.ragged_k = true;
  w.map_ws = map_ws;
  w.offsets = offsets;
  w.num_groups = groups;
  w.max_rows = rows;
  w.status = status;
  // dW2_e [D,F] = dYw_e^T h_e
  w.a[0] = act(dyw, rows, D);
  w.b[0] = act(h, rows, F);
  w.m_size = D;
  w.n_size = F;
  w.out0 = dw2;
  w.ld_out = F;
  w.group_stride_out = static_cast<int64_t>(D) * F;
  MOE_CUDA(gemm(moe::TIMING_WGRAD, w, st));

  // dx_rows = da1 w1_e + da3 w3_e (the dYw buffer may be reused as dx_rows)
  GemmArgs d;
  d.w8 = w8;
  d.w8_scale[0] = s1;
  d.w8_scale[1] = s3;
  d.epi = moe::EPI_BF16;
  d.b_mn = true;
  d.a[0] = act(da1, rows, F);
  d.a[1] = act(da3, rows, F);
  d.b[0] = wstack(w1, groups, F, D);  // B[n=d, k=f], d contiguous
  d.b[1] = wstack(w3, groups, F, D);
  d.k0 = F;
  d.k1 = F;
  d.offsets = offsets;
  d.num_groups = groups;
  d.max_rows = rows;
  d.n_size = D;
  d.out0 = dx_rows;
  d.ld_out = D;
  d.status = status;
  MOE_CUDA(gemm(moe::TIMING_DGRAD, d, st));

  // dW1_e [F,D] = da1_e^T x_e, dW3_e = da3_e^T x_e
  w.a[0] = act(da1, rows, F);
  w.b[0] = act(a_in, rows, D);
  w.m_size = F;
  w.n_size = D;
  w.out0 = dw1;
  w.ld_out = D;
  w.group_stride_out = static_cast<int64_t>(F) * D;
  MOE_CUDA(gemm(moe::TIMING_WGRAD, w, st));
  w.a[0] = act(da3, rows, F);
  w.out0 = dw3;
  MOE_CUDA(gemm(moe::TIMING_WGRAD, w, st));
  return MOE_OK;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device status error";
  }
  return "unknown";
}

moe_status_t moe_workspace_size(const moe_desc_t* d, size_t* fwd_bytes, size_t* bwd_bytes) {
  MOE_TRY(check_desc(d));
  const WsLayout L = layout(*d);
  if (fwd_bytes) *fwd_bytes = L.fwd_end;
  if (bwd_bytes) *bwd_bytes = L.total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kAlign || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  // all of it: the status block and the permute's look-back words start at zero
  MOE_CUDA(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_get_device_status(const void* ws, int32_t* status_host, void* stream) {
  if (!ws || !status_host) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  MOE_CUDA(cudaMemcpy(status_host, ws, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

// The ordered sum of the logits' ks contraction slices (ks == 1: part is the
// logits), top-K, histogram and scan in one launch.
static moe_status_t route_tail(const moe_desc_t* d, const float* part, int ks, float* logits, const float* bias,
                               int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, void* ws,
                               const WsLayout& L, cudaStream_t st) {
  moe::RouteShape rs{d->n_tok, d->n_exp, d->top_k, d->gate};
  int32_t* status = at<int32_t>(ws, L.status);
  return cuda_status(moe::launch_topk_scan(rs, part, ks, logits, d->use_bias ? bias : nullptr, topk_idx, topk_w,
                                           counts, offsets, at<int32_t>(ws, L.racc), status + kTicketWord, status,
                                           st));
}

moe_status_t moe_route(const moe_desc_t* d, const void* x, const void* w_gate, const float* bias, float* logits,
                       int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, void* ws,
                       size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_route");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!all16({x, w_gate, logits}) || !topk_idx || !topk_w || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (d->use_bias && !bias) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* dense = at<int32_t>(ws, L.dense_off);
  if (d->n_tok == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->n_exp, st));
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->n_exp + 1), st));
  }
  if (d->n_exp <= 32) {
    // one launch: logits on the warp-level MMA, top-K, histogram, scan (the
    // ticket counter lives in the status block moe_workspace_init clears)
    moe::RouteShape rs{d->n_tok, d->n_exp, d->top_k, d->gate};
    return cuda_status(moe::launch_router_fused(rs, d->d_model, x, w_gate, d->use_bias ? bias : nullptr, logits,
                                                topk_idx, topk_w, counts, offsets, status + kRouterAccWord,
                                                status + kTicketWord, status, st));
  }
  MOE_CUDA(moe::launch_dense_offsets(dense, d->n_tok, st));
  GemmArgs g;
  g.epi = moe::EPI_F32;
  g.block_n = d->n_exp <= 32 ? 32 : 256;
  g.a[0] = act(x, d->n_tok, d->d_model);
  g.b[0] = wstack(w_gate, 1, d->n_exp, d->d_model);
  g.k0 = d->d_model;
  g.offsets = dense;
  g.num_groups = 1;
  g.max_rows = d->n_tok;
  g.n_size = d->n_exp;
  g.ld_out = d->n_exp;
  g.status = status;
  // more CTAs than 128-token tiles: contraction slices into the workspace, then their ordered sum
  const int64_t tiles = (static_cast<int64_t>(d->n_tok) + 127) / 128 * ((d->n_exp + g.block_n - 1) / g.block_n);
  const int64_t ne = static_cast<int64_t>(d->n_tok) * d->n_exp;
  const int want = static_cast<int>(std::min<int64_t>(kGateSlices, moe::num_sms() / std::max<int64_t>(tiles, 1)));
  g.ksplit = ne % 4 == 0 ? moe::gemm_ksplit(d->d_model, want) : 1;
  float* part = at<float>(ws, L.gpart);
  g.out0 = g.ksplit > 1 ? static_cast<void*>(part) : static_cast<void*>(logits);
  MOE_CUDA(gemm(moe::TIMING_GATE, g, st));
  if (g.ksplit > 1) return route_tail(d, part, g.ksplit, logits, bias, topk_idx, topk_w, counts, offsets, ws, L, st);
  return route_tail(d, logits, 1, nullptr, bias, topk_idx, topk_w, counts, offsets, ws, L, st);
}

moe_status_t moe_route_from_logits(const moe_desc_t* d, const float* logits, const float* bias,
                                   int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                   void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_route_from_logits");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!logits || !topk_idx || !topk_w || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (d->use_bias && !bias) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  if (d->n_tok == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->n_exp, st));
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->n_exp + 1), st));
  }
  return route_tail(d, logits, 1, nullptr, bias, topk_idx, topk_w, counts, offsets, ws, L, st);
}

// moe_route_permute's scratch words, 128-byte aligned inside their region
// (the region has 128 bytes to spare; the workspace itself is 16-byte aligned)
static int32_t* rp_words(void* ws, const WsLayout& L) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(static_cast<char*>(ws) + L.rp_hist);
  return reinterpret_cast<int32_t*>((a + 127) & ~uintptr_t(127));
}

moe_status_t moe_route_permute(const moe_desc_t* d, const void* x, const void* w_gate, const float* bias,
                               float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                               int32_t* row_of_copy, int32_t* copy_of_row, void* x_perm, void* ws, size_t ws_bytes,
                               void* stream) {
  MOE_RANGE("moe_route_permute");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (d->n_exp > 32 || d->precision == 1) return MOE_ERR_INVALID_ARG;
  if (!all16({x, w_gate, logits, x_perm}) || !topk_idx || !topk_w || !counts || !offsets || !row_of_copy ||
      !copy_of_row)
    return MOE_ERR_INVALID_ARG;
  if (d->use_bias && !bias) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d->n_tok == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->n_exp, st));
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->n_exp + 1), st));
  }
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  moe::RouteShape rs{d->n_tok, d->n_exp, d->top_k, d->gate};
  return cuda_status(moe::launch_route_permute(rs, d->d_model, x, w_gate, d->use_bias ? bias : nullptr, logits,
                                               topk_idx, topk_w, counts, offsets, row_of_copy, copy_of_row, x_perm,
                                               rp_words(ws, L), status, st));
}

moe_status_t moe_permute(const moe_desc_t* d, const void* x, const int32_t* topk_idx, const int32_t* offsets,
                         int32_t* row_of_copy, int32_t* copy_of_row, void* x_perm, void* ws, size_t ws_bytes,
                         void* stream) {
  MOE_RANGE("moe_permute");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!all16({x, x_perm}) || !topk_idx || !offsets || !row_of_copy || !copy_of_row) return MOE_ERR_INVALID_ARG;
  if (d->n_tok == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  if (moe::permute_single_pass_look_words(d->n_tok, d->n_exp) <= static_cast<int64_t>(kLookWords))
    return cuda_status(moe::launch_permute_single_pass(d->n_tok, d->n_exp, d->top_k, d->d_model, topk_idx, offsets,
                                                       x, row_of_copy, copy_of_row, x_perm,
                                                       at<unsigned long long>(ws, L.look),
                                                       status + kPermuteCtlWord, status, st));
  MOE_CUDA(moe::launch_permute_maps(d->n_tok, d->n_exp, d->top_k, topk_idx, offsets, at<int32_t>(ws, L.blk_counts),
                                    at<int32_t>(ws, L.blk_base), row_of_copy, copy_of_row, status, st));
  return cuda_status(moe::launch_permute_rows(d->n_tok, d->d_model, d->top_k, x, row_of_copy, x_perm, st));
}

moe_status_t moe_grouped_ffn(const moe_desc_t* d, const void* x_perm, const int32_t* offsets, const void* x,
                             const moe_expert_weights_t* w, const moe_ffn_saved_t* saved, void* y_perm,
                             void* y_shared, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_grouped_ffn");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (d->precision != 0) return MOE_ERR_UNSUPPORTED;   // MXFP8 operands: moe_grouped_ffn_mxfp8
  if (!w || !saved || !offsets) return MOE_ERR_INVALID_ARG;
  if (!all16({x_perm, w->w1, w->w3, w->w2, saved->h, y_perm})) return MOE_ERR_INVALID_ARG;
  if ((saved->a1 && !aligned16(saved->a1)) || (saved->a3 && !aligned16(saved->a3))) return MOE_ERR_INVALID_ARG;
  if (d->n_shared) {
    if (!all16({x, w->ws1, w->ws3, w->ws2, saved->hs, y_shared})) return MOE_ERR_INVALID_ARG;
    if ((saved->a1s && !aligned16(saved->a1s)) || (saved->a3s && !aligned16(saved->a3s)))
      return MOE_ERR_INVALID_ARG;
  }
  if (d->n_tok == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  const int64_t R = static_cast<int64_t>(d->n_tok) * d->top_k;
  MOE_TRY(ffn_pair(x_perm, R, d->d_model, d->d_ff, d->n_exp, offsets, w->w1, w->w3, w->w2, saved->h, saved->a1,
                   saved->a3, y_perm, status, st));
  if (d->n_shared) {
    int32_t* dense = at<int32_t>(ws, L.dense_off);
    MOE_CUDA(moe::launch_dense_offsets(dense, d->n_tok, st));
    MOE_TRY(ffn_pair(x, d->n_tok, d->d_model, d->d_ff_shared, 1, dense, w->ws1, w->ws3, w->ws2, saved->hs,
                     saved->a1s, saved->a3s, y_shared, status, st));
  }
  return MOE_OK;
}

moe_status_t moe_permute_maps(const moe_desc_t* d, const int32_t* topk_idx, const int32_t* offsets,
                              int32_t* row_of_copy, int32_t* copy_of_row, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_permute_maps");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!topk_idx || !offsets || !row_of_copy || !copy_of_row) return MOE_ERR_INVALID_ARG;
  if (d->n_tok == 0) return MOE_OK;
  const WsLayout L = layout(*d);
  return cuda_status(moe::launch_permute_maps(d->n_tok, d->n_exp, d->top_k, topk_idx, offsets,
                                              at<int32_t>(ws, L.blk_counts), at<int32_t>(ws, L.blk_base),
                                              row_of_copy, copy_of_row, at<int32_t>(ws, L.status),
                                              static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_ffn_gather(const moe_desc_t* d, const void* x, const int32_t* copy_of_row,
                                    const int32_t* offsets, const moe_expert_weights_t* w, const moe_ffn_saved_t* saved,
                                    void* y_perm, void* y_shared, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_grouped_ffn_gather");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (d->precision != 0) return MOE_ERR_UNSUPPORTED;
  if (!w || !saved || !offsets || !copy_of_row) return MOE_ERR_INVALID_ARG;
  if (!all16({x, w->w1, w->w3, w->w2, saved->h, y_perm})) return MOE_ERR_INVALID_ARG;
  if ((saved->a1 && !aligned16(saved->a1)) || (saved->a3 && !aligned16(saved->a3))) return MOE_ERR_INVALID_ARG;
  if (d->n_shared) {
    if (!all16({w->ws1, w->ws3, w->ws2, saved->hs, y_shared})) return MOE_ERR_INVALID_ARG;
    if ((saved->a1s && !aligned16(saved->a1s)) || (saved->a3s && !aligned16(saved->a3s)))
      return MOE_ERR_INVALID_ARG;
  }
  if (d->n_tok == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  const int64_t R = static_cast<int64_t>(d->n_tok) * d->top_k;
  MOE_TRY(ffn_pair(x, R, d->d_model, d->d_ff, d->n_exp, offsets, w->w1, w->w3, w->w2, saved->h, saved->a1,
                   saved->a3, y_perm, status, st, nullptr, nullptr, nullptr, copy_of_row, d->top_k, d->n_tok));
  if (d->n_shared) {
    int32_t* dense = at<int32_t>(ws, L.dense_off);
    MOE_CUDA(moe::launch_dense_offsets(dense, d->n_tok, st));
    MOE_TRY(ffn_pair(x, d->n_tok, d->d_model, d->d_ff_shared, 1, dense, w->ws1, w->ws3, w->ws2, saved->hs,
                     saved->a1s, saved->a3s, y_shared, status, st));
  }
  return MOE_OK;
}

moe_status_t moe_combine(const moe_desc_t* d, const void* y_perm, const int32_t* row_of_copy, const float* topk_w,
                         const void* y_shared, void* out, void* stream) {
  MOE_RANGE("moe_combine");
  MOE_TRY(check_desc(d));
  if (!all16({y_perm, out}) || !row_of_copy || !topk_w) return MOE_ERR_INVALID_ARG;
  if (y_shared && !aligned16(y_shared)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_combine(d->n_tok, d->d_model, d->top_k, y_perm, row_of_copy, topk_w, y_shared, out,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// The layer backward (moe_backward); with FP8 weights (q non-NULL) the data
// gradients read the E4M3 weight codes w1, w3, w2 with their tile scales.
moe_status_t backward_impl(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_t* w,
                           const moe_expert_weights_mx_t* q, const moe_fwd_state_t* s, const void* dy,
                           const moe_grads_t* g, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_ws(*d, ws, ws_bytes, true));
  if (!w || !s || !g) return MOE_ERR_INVALID_ARG;
  if (!all16({w_gate, w->w1, w->w3, w->w2, s->x, s->x_perm, s->a1, s->a3, s->h, s->y_perm, dy, g->dx, g->dw_gate,
              g->dw1, g->dw3, g->dw2}))
    return MOE_ERR_INVALID_ARG;
  if (!s->logits || !s->topk_idx || !s->topk_w || !s->offsets || !s->row_of_copy || !s->copy_of_row)
    return MOE_ERR_INVALID_ARG;
  if (d->n_shared && !all16({w->ws1, w->ws3, w->ws2, s->a1s, s->a3s, s->hs, g->dws1, g->dws3, g->dws2}))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  const int N = d->n_tok, D = d->d_model, F = d->d_ff, E = d->n_exp, K = d->top_k;
  const int64_t R = static_cast<int64_t>(N) * K;
  if (N == 0) {
    MOE_CUDA(cudaMemsetAsync(g->dw_gate, 0, sizeof(float) * E * D, st));
    MOE_CUDA(cudaMemsetAsync(g->dw1, 0, sizeof(float) * E * F * D, st));
    MOE_CUDA(cudaMemsetAsync(g->dw3, 0, sizeof(float) * E * F * D, st));
    MOE_CUDA(cudaMemsetAsync(g->dw2, 0, sizeof(float) * E * F * D, st));
    if (d->n_shared) {
      const size_t fs = d->d_ff_shared;
      MOE_CUDA(cudaMemsetAsync(g->dws1, 0, sizeof(float) * fs * D, st));
      MOE_CUDA(cudaMemsetAsync(g->dws3, 0, sizeof(float) * fs * D, st));
      MOE_CUDA(cudaMemsetAsync(g->dws2, 0, sizeof(float) * fs * D, st));
    }
    return MOE_OK;
  }
  int32_t* status = at<int32_t>(ws, L.status);
  float* dl = g->dlogits ? g->dlogits : at<float>(ws, L.dl);
  float* dg = g->dg ? g->dg : at<float>(ws, L.dg);
  void* dyw = at<void>(ws, L.dyw);
  void* da1 = at<void>(ws, L.da1);
  void* da3 = at<void>(ws, L.da3);

  MOE_CUDA(moe::launch_combine_bwd(N, D, K, d->gate, dy, s->y_perm, s->row_of_copy, s->topk_w, s->logits, E,
                                   s->topk_idx, dyw, dg, dl, st));
  // routed experts; dx_perm overwrites dYw once its last reader is done
  auto sc = [&](const void* p_) { return q ? static_cast<const float*>(p_) : nullptr; };
  MOE_TRY(ffn_pair_bwd(dyw, s->x_perm, s->a1, s->a3, s->h, R, D, F, E, s->offsets, w->w1, w->w3, w->w2, da1, da3,
                       dyw, g->dw1, g->dw3, g->dw2, status, st, map_scratch(ws, L), sc(q ? q->w1_scale : nullptr),
                       sc(q ? q->w3_scale : nullptr), sc(q ? q->w2_scale : nullptr)));
  void* dxs = nullptr;
  if (d->n_shared) {
    int32_t* dense = at<int32_t>(ws, L.dense_off);
    MOE_CUDA(moe::launch_dense_offsets(dense, N, st));
    dxs = at<void>(ws, L.dxs);
    MOE_TRY(ffn_pair_bwd(dy, s->x, s->a1s, s->a3s, s->hs, N, D, d->d_ff_shared, 1, dense, w->ws1, w->ws3, w->ws2,
                         at<void>(ws, L.da1s), at<void>(ws, L.da3s), dxs, g->dws1, g->dws3, g->dws2, status, st,
                         map_scratch(ws, L), sc(q ? q->ws1_scale : nullptr), sc(q ? q->ws3_scale : nullptr),
                         sc(q ? q->ws2_scale : nullptr)));
  }
  if (s->offsets_full && s->copy_of_row_full)   // capacity mode: every copy, x gathered in dropless order
    MOE_CUDA(moe::launch_dwgate(N, K, E, D, s->offsets_full, s->copy_of_row_full, dl, s->x, K,
                                at<float>(ws, L.dwg), g->dw_gate, st));
  else
    MOE_CUDA(moe::launch_dwgate(N, K, E, D, s->offsets, s->copy_of_row, dl, s->x_perm, 0, at<float>(ws, L.dwg),
                                g->dw_gate, st));
  MOE_CUDA(moe::launch_unpermute_dx(N, D, K, dyw, s->row_of_copy, dl, s->topk_idx, w_gate, dxs, g->dx, st));
  return MOE_OK;
}
}  // namespace

extern "C" {

moe_status_t moe_backward(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_t* w,
                          const moe_fwd_state_t* s, const void* dy, const moe_grads_t* g, void* ws,
                          size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_backward");
  MOE_TRY(check_desc(d));
  if (d->precision != 0) return MOE_ERR_UNSUPPORTED;   // bf16 operands; moe_backward_mxfp8 / _fp8w otherwise
  return backward_impl(d, w_gate, w, nullptr, s, dy, g, ws, ws_bytes, stream);
}

moe_status_t moe_backward_fp8w(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_mx_t* wq,
                               const moe_fwd_state_t* s, const void* dy, const moe_grads_t* g, void* ws,
                               size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_backward_fp8w");
  MOE_TRY(check_desc(d));
  if (d->precision != 2 || !wq) return MOE_ERR_INVALID_ARG;
  if (!wq->w1_scale || !wq->w3_scale || !wq->w2_scale) return MOE_ERR_INVALID_ARG;
  if (d->n_shared && (!wq->ws1_scale || !wq->ws3_scale || !wq->ws2_scale)) return MOE_ERR_INVALID_ARG;
  const moe_expert_weights_t w{wq->w1, wq->w3, wq->w2, wq->ws1, wq->ws3, wq->ws2};
  return backward_impl(d, w_gate, &w, wq, s, dy, g, ws, ws_bytes, stream);
}

moe_status_t moe_quantize_mxfp8(const void* src, int64_t groups, int64_t rows, int64_t cols, void* codes,
                                void* scales, int64_t scale_ld, void* stream) {
  MOE_RANGE("moe_quantize_mxfp8");
  if (groups <= 0 || rows <= 0 || cols <= 0 || cols % 32 || scale_ld < rows || scale_ld % 16) return MOE_ERR_INVALID_ARG;
  if (!all16({src, codes, scales})) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_mx_quant_rows(src, nullptr, 1, groups * rows, static_cast<int>(cols), rows, scale_ld,
                                               static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales),
                                               static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_permute_mxfp8(const moe_desc_t* d, const void* x, const int32_t* topk_idx, const int32_t* offsets,
                               int32_t* row_of_copy, int32_t* copy_of_row, void* xq_perm, void* xs_perm,
                               void* xq_tok, void* xs_tok, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_permute_mxfp8");
  MOE_TRY(check_desc(d));
  if (d->precision != 1) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!all16({x, xq_perm, xs_perm}) || !topk_idx || !offsets || !row_of_copy || !copy_of_row)
    return MOE_ERR_INVALID_ARG;
  if (xq_tok && !all16({xq_tok, xs_tok})) return MOE_ERR_INVALID_ARG;
  if (d->n_tok == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  const int64_t R = static_cast<int64_t>(d->n_tok) * d->top_k;
  int32_t* status = at<int32_t>(ws, L.status);
  if (moe::permute_single_pass_look_words(d->n_tok, d->n_exp) <= static_cast<int64_t>(kLookWords))
    return cuda_status(moe::launch_permute_single_pass_mxfp8(
        d->n_tok, d->n_exp, d->top_k, d->d_model, topk_idx, offsets, x, row_of_copy, copy_of_row,
        static_cast<uint8_t*>(xq_perm), static_cast<uint8_t*>(xs_perm), moe::mx_scale_ld(R),
        static_cast<uint8_t*>(xq_tok), static_cast<uint8_t*>(xq_tok ? xs_tok : nullptr), moe::mx_scale_ld(d->n_tok),
        at<unsigned long long>(ws, L.look), status + kPermuteCtlWord, status, st));
  MOE_CUDA(moe::launch_permute_maps(d->n_tok, d->n_exp, d->top_k, topk_idx, offsets, at<int32_t>(ws, L.blk_counts),
                                    at<int32_t>(ws, L.blk_base), row_of_copy, copy_of_row, status, st));
  MOE_CUDA(moe::launch_mx_quant_rows(x, copy_of_row, d->top_k, R, d->d_model, R, moe::mx_scale_ld(R),
                                     static_cast<uint8_t*>(xq_perm), static_cast<uint8_t*>(xs_perm), st));
  if (xq_tok)
    MOE_CUDA(moe::launch_mx_quant_rows(x, nullptr, 1, d->n_tok, d->d_model, d->n_tok, moe::mx_scale_ld(d->n_tok),
                                       static_cast<uint8_t*>(xq_tok), static_cast<uint8_t*>(xs_tok), st));
  return MOE_OK;
}

namespace {
// MXFP8 SwiGLU FFN of one expert set: GEMM1 (w1|w3, SwiGLU, h quantised) then GEMM2.
moe_status_t ffn_pair_mx(const void* aq, const void* as, int64_t rows, int D, int F, int groups,
                         const int32_t* offsets, const void* w1, const void* w1s, const void* w3, const void* w3s,
                         const void* w2, const void* w2s, void* hq, void* hs, void* h, void* a1, void* a3, void* y,
                         int32_t* status, cudaStream_t st) {
  GemmArgs g1;
  g1.quant = true;
  g1.epi = moe::EPI_SWIGLU_FWD_Q;
  g1.qa[0] = moe::MxOperand{aq, as, rows, D, 1, moe::mx_scale_ld(rows)};
  g1.qb[0] = moe::MxOperand{w1, w1s, F, D, groups, F};
  g1.qb[1] = moe::MxOperand{w3, w3s, F, D, groups, F};
  g1.b_dual_n = true;
  g1.k0 = D;
  g1.offsets = offsets;
  g1.num_groups = groups;
  g1.max_rows = rows;
  g1.n_size = F;
  g1.out0 = hq;
  g1.out1 = hs;
  g1.out2 = h;
  g1.out3 = a1;
  g1.out4 = a3;
  g1.s_ld = moe::mx_scale_ld(rows);
  g1.ld_out = F;
  g1.status = status;
  MOE_CUDA(gemm(moe::TIMING_FFN_FWD, g1, st));
  GemmArgs g2;
  g2.quant = true;
  g2.epi = moe::EPI_BF16;
  g2.qa[0] = moe::MxOperand{hq, hs, rows, F, 1, moe::mx_scale_ld(rows)};
  g2.qb[0] = moe::MxOperand{w2, w2s, D, F, groups, D};
  g2.k0 = F;
  g2.offsets = offsets;
  g2.num_groups = groups;
  g2.max_rows = rows;
  g2.n_size = D;
  g2.out0 = y;
  g2.ld_out = D;
  g2.status = status;
  MOE_CUDA(gemm(moe::TIMING_FFN_FWD, g2, st));
  return MOE_OK;
}
// Workspace scratch of one MXFP8 backward expert set.
struct MxBwdScratch {
  uint8_t *q_dy, *q_dys, *q_da1, *q_da1s, *q_da3, *q_da3s;
  int32_t* pad;
  int64_t rp;
  uint8_t *t_d0, *t_d0s, *t_d1, *t_d1s, *t_f0, *t_f0s, *t_f1, *t_f1s;
};

// MXFP8 backward of one expert set (moe_backward_mxfp8): dgrad through w2
// with the SwiGLU derivative, dW2, dgrad through w1|w3, dW1, dW3.  x_rows is
// the expert set's input, row r read as x_rows[gather[r] / gather_k] when
// `gather` is given.  dx_rows may alias dyw.
moe_status_t ffn_pair_bwd_mx(const void* dyw, const void* x_rows, const int32_t* gather, int gather_k,
                             const void* a1, const void* a3, const void* h, int64_t rows, int D, int F, int groups,
                             const int32_t* offsets, const void* w1t, const void* w1ts, const void* w3t,
                             const void* w3ts, const void* w2t, const void* w2ts, void* da1, void* da3,
                             void* dx_rows, float* dw1, float* dw3, float* dw2, const MxBwdScratch& q,
                             int32_t* status, cudaStream_t st, bool dyw_quantized = false) {
  const int64_t ldr = moe::mx_scale_ld(rows);
  // dYw row-wise along D (unless the combine backward already wrote these
  // codes); dh = dYw w2 with the SwiGLU derivative -> da1, da3 (bf16)
  if (!dyw_quantized)
    MOE_CUDA(moe::launch_mx_quant_rows(dyw, nullptr, 1, rows, D, rows, ldr, q.q_dy, q.q_dys, st));
  GemmArgs g;
  g.quant = true;
  g.epi = moe::EPI_SWIGLU_BWD;
  g.qa[0] = moe::MxOperand{q.q_dy, q.q_dys, rows, D, 1, ldr};
  g.qb[0] = moe::MxOperand{w2t, w2ts, F, D, groups, F};
  g.k0 = D;
  g.offsets = offsets;
  g.num_groups = groups;
  g.max_rows = rows;
  g.n_size = F;
  g.in0 = a1;
  g.in1 = a3;
  g.out0 = da1;
  g.out1 = da3;
  g.ld_out = F;
  g.status = status;
  MOE_CUDA(gemm(moe::TIMING_DGRAD, g, st));

  // weight-gradient operands: blocks of 32 tokens per expert, transposed
  MOE_CUDA(moe::launch_pad_offsets(offsets, groups, q.pad, st));
  auto tquant = [&](const void* src, const int32_t* gat, int gk, int cols, uint8_t* codes, uint8_t* scales) {
    return moe::launch_mx_quant_cols_t(src, 1, rows, cols, gat, gk, offsets, q.pad, groups, q.rp, codes, ld16(cols),
                                       scales, st);
  };
  MOE_CUDA(tquant(dyw, nullptr, 1, D, q.t_d0, q.t_d0s));
  MOE_CUDA(tquant(h, nullptr, 1, F, q.t_f0, q.t_f0s));
  GemmArgs w;
  w.quant = true;
  w.epi = moe::EPI_F32;
  w.ragged_k = true;
  w.offsets = q.pad;
  w.num_groups = groups;
  w.max_rows = rows;
  w.status = status;
  // dW2_e [D,F] = dYw_e^T h_e
  w.qa[0] = moe::MxOperand{q.t_d0, q.t_d0s, D, q.rp, 1, ld16(D)};
  w.qb[0] = moe::MxOperand{q.t_f0, q.t_f0s, F, q.rp, 1, ld16(F)};
  w.m_size = D;
  w.n_size = F;
  w.out0 = dw2;
  w.ld_out = F;
  w.group_stride_out = static_cast<int64_t>(D) * F;
  MOE_CUDA(gemm(moe::TIMING_WGRAD, w, st));

  // da1, da3 row-wise along F; dx_rows = da1 w1 + da3 w3 (dYw is no longer read)
  MOE_CUDA(moe::launch_mx_quant_rows(da1, nullptr, 1, rows, F, rows, ldr, q.q_da1, q.q_da1s, st));
  MOE_CUDA(moe::launch_mx_quant_rows(da3, nullptr, 1, rows, F, rows, ldr, q.q_da3, q.q_da3s, st));
  GemmArgs d;
  d.quant = true;
  d.epi = moe::EPI_BF16;
  d.qa[0] = moe::MxOperand{q.q_da1, q.q_da1s, rows, F, 1, ldr};
  d.qa[1] = moe::MxOperand{q.q_da3, q.q_da3s, rows, F, 1, ldr};
  d.qb[0] = moe::MxOperand{w1t, w1ts, D, F, groups, D};
  d.qb[1] = moe::MxOperand{w3t, w3ts, D, F, groups, D};
  d.k0 = F;
  d.k1 = F;
  d.offsets = offsets;
  d.num_groups = groups;
  d.max_rows = rows;
  d.n_size = D;
  d.out0 = dx_rows;
  d.ld_out = D;
  d.status = status;
  MOE_CUDA(gemm(moe::TIMING_DGRAD, d, st));

  // dW1_e [F,D] = da1_e^T x_e, dW3_e = da3_e^T x_e
  MOE_CUDA(tquant(da1, nullptr, 1, F, q.t_f0, q.t_f0s));
  MOE_CUDA(tquant(da3, nullptr, 1, F, q.t_f1, q.t_f1s));
  MOE_CUDA(tquant(x_rows, gather, gather_k, D, q.t_d1, q.t_d1s));
  w.qa[0] = moe::MxOperand{q.t_f0, q.t_f0s, F, q.rp, 1, ld16(F)};
  w.qb[0] = moe::MxOperand{q.t_d1, q.t_d1s, D, q.rp, 1, ld16(D)};
  w.m_size = F;
  w.n_size = D;
  w.out0 = dw1;
  w.ld_out = D;
  w.group_stride_out = static_cast<int64_t>(F) * D;
  MOE_CUDA(gemm(moe::TIMING_WGRAD, w, st));
  w.qa[0] = moe::MxOperand{q.t_f1, q.t_f1s, F, q.rp, 1, ld16(F)};
  w.out0 = dw3;
  MOE_CUDA(gemm(moe::TIMING_WGRAD, w, st));
  return MOE_OK;
}
}  // namespace

moe_status_t moe_grouped_ffn_mxfp8(const moe_desc_t* d, const void* xq_perm, const void* xs_perm,
                                   const int32_t* offsets, const void* xq_tok, const void* xs_tok,
                                   const moe_expert_weights_mx_t* w, const moe_ffn_saved_t* saved, void* y_perm,
                                   void* y_shared, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_grouped_ffn_mxfp8");
  MOE_TRY(check_desc(d));
  if (d->precision != 1) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!w || !offsets || !all16({xq_perm, xs_perm, w->w1, w->w1_scale, w->w3, w->w3_scale, w->w2, w->w2_scale, y_perm}))
    return MOE_ERR_INVALID_ARG;
  moe_ffn_saved_t sv{};
  if (saved) sv = *saved;
  for (const void* q : {sv.a1, sv.a3, sv.h, sv.a1s, sv.a3s, sv.hs})
    if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (d->n_shared && !all16({xq_tok, xs_tok, w->ws1, w->ws1_scale, w->ws3, w->ws3_scale, w->ws2, w->ws2_scale,
                             y_shared}))
    return MOE_ERR_INVALID_ARG;
  if (d->n_tok == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  const int64_t R = static_cast<int64_t>(d->n_tok) * d->top_k;
  MOE_TRY(ffn_pair_mx(xq_perm, xs_perm, R, d->d_model, d->d_ff, d->n_exp, offsets, w->w1, w->w1_scale, w->w3,
                      w->w3_scale, w->w2, w->w2_scale, at<void>(ws, L.hq), at<void>(ws, L.hs), sv.h, sv.a1, sv.a3,
                      y_perm, status, st));
  if (d->n_shared) {
    int32_t* dense = at<int32_t>(ws, L.dense_off);
    MOE_CUDA(moe::launch_dense_offsets(dense, d->n_tok, st));
    MOE_TRY(ffn_pair_mx(xq_tok, xs_tok, d->n_tok, d->d_model, d->d_ff_shared, 1, dense, w->ws1, w->ws1_scale, w->ws3,
                        w->ws3_scale, w->ws2, w->ws2_scale, at<void>(ws, L.hq_sh), at<void>(ws, L.hs_sh), sv.hs,
                        sv.a1s, sv.a3s, y_shared, status, st));
  }
  return MOE_OK;
}

moe_status_t moe_quantize_mxfp8_t(const void* src, int64_t groups, int64_t rows, int64_t cols, void* codes,
                                  void* scales, int64_t scale_ld, void* stream) {
  MOE_RANGE("moe_quantize_mxfp8_t");
  if (!all16({src, codes}) || !scales || groups < 1 || rows <= 0 || cols <= 0 || rows % 32 || cols % 8 ||
      scale_ld < cols || scale_ld % 16 || cols > (int64_t{1} << 30))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_mx_quant_cols_t(src, groups, rows, static_cast<int>(cols), nullptr, 1, nullptr,
                                                 nullptr, 1, rows, static_cast<uint8_t*>(codes), scale_ld,
                                                 static_cast<uint8_t*>(scales), static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_backward_mxfp8(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_mx_t* wt,
                                const moe_fwd_state_t* s, const void* dy, const moe_grads_t* g, void* ws,
                                size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_backward_mxfp8");
  MOE_TRY(check_desc(d));
  if (d->precision != 1) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(*d, ws, ws_bytes, true));
  if (!wt || !s || !g) return MOE_ERR_INVALID_ARG;
  if (!all16({w_gate, wt->w1, wt->w1_scale, wt->w3, wt->w3_scale, wt->w2, wt->w2_scale, s->x, s->a1, s->a3, s->h,
              s->y_perm, dy, g->dx, g->dw_gate, g->dw1, g->dw3, g->dw2}))
    return MOE_ERR_INVALID_ARG;
  if (!s->logits || !s->topk_idx || !s->topk_w || !s->offsets || !s->row_of_copy || !s->copy_of_row)
    return MOE_ERR_INVALID_ARG;
  if (d->n_shared && !all16({wt->ws1, wt->ws1_scale, wt->ws3, wt->ws3_scale, wt->ws2, wt->ws2_scale, s->a1s,
                             s->a3s, s->hs, g->dws1, g->dws3, g->dws2}))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  const int N = d->n_tok, D = d->d_model, F = d->d_ff, E = d->n_exp, K = d->top_k;
  const int64_t R = static_cast<int64_t>(N) * K;
  if (N == 0) {
    MOE_CUDA(cudaMemsetAsync(g->dw_gate, 0, sizeof(float) * E * D, st));
    MOE_CUDA(cudaMemsetAsync(g->dw1, 0, sizeof(float) * E * F * D, st));
    MOE_CUDA(cudaMemsetAsync(g->dw3, 0, sizeof(float) * E * F * D, st));
    MOE_CUDA(cudaMemsetAsync(g->dw2, 0, sizeof(float) * E * F * D, st));
    if (d->n_shared) {
      const size_t fs = d->d_ff_shared;
      MOE_CUDA(cudaMemsetAsync(g->dws1, 0, sizeof(float) * fs * D, st));
      MOE_CUDA(cudaMemsetAsync(g->dws3, 0, sizeof(float) * fs * D, st));
      MOE_CUDA(cudaMemsetAsync(g->dws2, 0, sizeof(float) * fs * D, st));
    }
    return MOE_OK;
  }
  int32_t* status = at<int32_t>(ws, L.status);
  float* dl = g->dlogits ? g->dlogits : at<float>(ws, L.dl);
  float* dg = g->dg ? g->dg : at<float>(ws, L.dg);
  void* dyw = at<void>(ws, L.dyw);
  MxBwdScratch q{at<uint8_t>(ws, L.q_dy), at<uint8_t>(ws, L.q_dys), at<uint8_t>(ws, L.q_da1),
                 at<uint8_t>(ws, L.q_da1s), at<uint8_t>(ws, L.q_da3), at<uint8_t>(ws, L.q_da3s),
                 at<int32_t>(ws, L.pad), L.rp, at<uint8_t>(ws, L.t_d0), at<uint8_t>(ws, L.t_d0s),
                 at<uint8_t>(ws, L.t_d1), at<uint8_t>(ws, L.t_d1s), at<uint8_t>(ws, L.t_f0),
                 at<uint8_t>(ws, L.t_f0s), at<uint8_t>(ws, L.t_f1), at<uint8_t>(ws, L.t_f1s)};

  // dYw and, fused, its row-wise MXFP8 codes along D
  MOE_CUDA(moe::launch_combine_bwd(N, D, K, d->gate, dy, s->y_perm, s->row_of_copy, s->topk_w, s->logits, E,
                                   s->topk_idx, dyw, dg, dl, st, q.q_dy, q.q_dys, moe::mx_scale_ld(R)));
  // routed experts (x read in permuted order through copy_of_row); dx_perm overwrites dYw
  MOE_TRY(ffn_pair_bwd_mx(dyw, s->x, s->copy_of_row, K, s->a1, s->a3, s->h, R, D, F, E, s->offsets, wt->w1,
                          wt->w1_scale, wt->w3, wt->w3_scale, wt->w2, wt->w2_scale, at<void>(ws, L.da1),
                          at<void>(ws, L.da3), dyw, g->dw1, g->dw3, g->dw2, q, status, st, true));
  void* dxs = nullptr;
  if (d->n_shared) {
    int32_t* dense = at<int32_t>(ws, L.dense_off);
    MOE_CUDA(moe::launch_dense_offsets(dense, N, st));
    dxs = at<void>(ws, L.dxs);
    MxBwdScratch qs = q;
    qs.pad = at<int32_t>(ws, L.pad_sh);
    MOE_TRY(ffn_pair_bwd_mx(dy, s->x, nullptr, 1, s->a1s, s->a3s, s->hs, N, D, d->d_ff_shared, 1, dense, wt->ws1,
                            wt->ws1_scale, wt->ws3, wt->ws3_scale, wt->ws2, wt->ws2_scale, at<void>(ws, L.da1s),
                            at<void>(ws, L.da3s), dxs, g->dws1, g->dws3, g->dws2, qs, status, st));
  }
  const bool full = s->offsets_full && s->copy_of_row_full;
  MOE_CUDA(moe::launch_dwgate(N, K, E, D, full ? s->offsets_full : s->offsets,
                              full ? s->copy_of_row_full : s->copy_of_row, dl, s->x, K, at<float>(ws, L.dwg),
                              g->dw_gate, st));
  MOE_CUDA(moe::launch_unpermute_dx(N, D, K, dyw, s->row_of_copy, dl, s->topk_idx, w_gate, dxs, g->dx, st));
  return MOE_OK;
}

moe_status_t moe_permute_capacity(const moe_desc_t* d, const void* x, const int32_t* topk_idx,
                                  const int32_t* offsets, double capacity_factor, int32_t* row_of_copy_full,
                                  int32_t* copy_of_row_full, int32_t* kept_offsets, int32_t* row_of_copy,
                                  int32_t* copy_of_row, void* x_perm, int32_t* n_dropped, void* ws,
                                  size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_permute_capacity");
  MOE_TRY(check_desc(d));
  if (d->precision != 0) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!all16({x, x_perm}) || !topk_idx || !offsets || !row_of_copy_full || !copy_of_row_full || !kept_offsets ||
      !row_of_copy || !copy_of_row || !(capacity_factor >= 0.0))
    return MOE_ERR_INVALID_ARG;
  const double capd = std::ceil(capacity_factor * (static_cast<double>(d->n_tok) / d->n_exp * d->top_k) - 1e-9);
  if (capd > 2147483647.0) return MOE_ERR_INVALID_ARG;
  const int cap = capd > 0.0 ? static_cast<int>(capd) : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  if (d->n_tok == 0) {
    MOE_CUDA(cudaMemsetAsync(kept_offsets, 0, sizeof(int32_t) * (d->n_exp + 1), st));
    return n_dropped ? cuda_status(cudaMemsetAsync(n_dropped, 0, sizeof(int32_t), st)) : MOE_OK;
  }
  MOE_CUDA(moe::launch_permute_maps(d->n_tok, d->n_exp, d->top_k, topk_idx, offsets, at<int32_t>(ws, L.blk_counts),
                                    at<int32_t>(ws, L.blk_base), row_of_copy_full, copy_of_row_full,
                                    at<int32_t>(ws, L.status), st));
  MOE_CUDA(moe::launch_capacity_maps(d->n_tok, d->n_exp, d->top_k, topk_idx, offsets, row_of_copy_full, cap,
                                     kept_offsets, row_of_copy, copy_of_row, n_dropped, st));
  MOE_CUDA(moe::launch_permute_rows(d->n_tok, d->d_model, d->top_k, x, row_of_copy, x_perm, st));
  return MOE_OK;
}

moe_status_t moe_quantize_fp8_tile(const void* src, int64_t groups, int64_t rows, int64_t cols, void* codes,
                                   float* scales, void* stream) {
  MOE_RANGE("moe_quantize_fp8_tile");
  if (!src || !codes || !scales || groups < 1 || rows <= 0 || cols <= 0 || cols % 16 || !aligned16(src) ||
      !aligned16(codes))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_fp8_tile_quant(src, groups, rows, cols, static_cast<uint8_t*>(codes), scales,
                                                static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_ffn_fp8w(const moe_desc_t* d, const void* x_perm, const int32_t* offsets, const void* x,
                                  const moe_expert_weights_mx_t* wq, const moe_ffn_saved_t* saved, void* y_perm,
                                  void* y_shared, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_grouped_ffn_fp8w");
  MOE_TRY(check_desc(d));
  if (d->precision != 2) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!wq || !saved || !offsets) return MOE_ERR_INVALID_ARG;
  if (!all16({x_perm, wq->w1, wq->w3, wq->w2, saved->h, y_perm}) || !wq->w1_scale || !wq->w3_scale || !wq->w2_scale)
    return MOE_ERR_INVALID_ARG;
  if ((saved->a1 && !aligned16(saved->a1)) || (saved->a3 && !aligned16(saved->a3))) return MOE_ERR_INVALID_ARG;
  if (d->n_shared && (!all16({x, wq->ws1, wq->ws3, wq->ws2, saved->hs, y_shared}) || !wq->ws1_scale ||
                      !wq->ws3_scale || !wq->ws2_scale))
    return MOE_ERR_INVALID_ARG;
  if (d->n_tok == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout L = layout(*d);
  int32_t* status = at<int32_t>(ws, L.status);
  const int64_t R = static_cast<int64_t>(d->n_tok) * d->top_k;
  MOE_TRY(ffn_pair(x_perm, R, d->d_model, d->d_ff, d->n_exp, offsets, wq->w1, wq->w3, wq->w2, saved->h, saved->a1,
                   saved->a3, y_perm, status, st, static_cast<const float*>(wq->w1_scale),
                   static_cast<const float*>(wq->w3_scale), static_cast<const float*>(wq->w2_scale)));
  if (d->n_shared) {
    int32_t* dense = at<int32_t>(ws, L.dense_off);
    MOE_CUDA(moe::launch_dense_offsets(dense, d->n_tok, st));
    MOE_TRY(ffn_pair(x, d->n_tok, d->d_model, d->d_ff_shared, 1, dense, wq->ws1, wq->ws3, wq->ws2, saved->hs,
                     saved->a1s, saved->a3s, y_shared, status, st, static_cast<const float*>(wq->ws1_scale),
                     static_cast<const float*>(wq->ws3_scale), static_cast<const float*>(wq->ws2_scale)));
  }
  return MOE_OK;
}

moe_status_t moe_aux_loss(const moe_desc_t* d, const float* logits, const int32_t* counts, float coef, float* loss,
                          float* dlogits_aux, void* ws, size_t ws_bytes, void* stream) {
  MOE_RANGE("moe_aux_loss");
  MOE_TRY(check_desc(d));
  MOE_TRY(check_ws(*d, ws, ws_bytes, false));
  if (!logits || !counts || !loss) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d->n_tok == 0) return cuda_status(cudaMemsetAsync(loss, 0, sizeof(float), st));
  const WsLayout L = layout(*d);
  return cuda_status(moe::launch_aux_loss(logits, d->n_tok, d->n_exp, d->gate, counts, coef, at<float>(ws, L.aux),
                                          loss, dlogits_aux, st));
}

moe_status_t moe_monitor_stats(int32_t n_exp, const int32_t* counts_hist, int32_t n_hist, float* stats,
                               void* stream) {
  MOE_RANGE("moe_monitor_stats");
  if (n_exp < 1 || n_exp > 1024 || n_hist < 1 || !counts_hist || !stats) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_monitor(counts_hist, n_hist, n_exp, stats, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_update_bias(const moe_desc_t* d, const int32_t* counts, float* bias, float gamma, int32_t mode,
                             void* stream) {
  MOE_RANGE("moe_update_bias");
  MOE_TRY(check_desc(d));
  if (!counts || !bias || (mode != 0 && mode != 1)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      moe::launch_update_bias(counts, d->n_exp, bias, gamma, mode, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
