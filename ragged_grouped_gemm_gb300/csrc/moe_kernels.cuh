// Launchers of the memory-bound kernels of the MoE layer (router top-K,
// histogram, scan, permute, combine and their backward counterparts).
// All launches are asynchronous on the given stream and read group sizes
// only on the device.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

struct RouteShape {
  int n_tok, n_exp, top_k;
  int gate;      // 0 softmax, 1 sigmoid
};

// The whole router of a layer with E <= 32 in one launch: logits (warp-level
// tensor-core MMA, fp32), then top-K, weights, counts and offsets as
// launch_topk_scan.  acc: E int32 and ticket: one int32, all zero
// before the launch (the kernel leaves them zero).  D must be a multiple of 32.
cudaError_t launch_router_fused(const RouteShape& s, int d, const void* x, const void* w_gate, const float* bias,
                                float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                int32_t* acc, int32_t* ticket, int32_t* status, cudaStream_t st);
// launch_router_fused and then the permute of the same tokens in one
// cooperative launch (E <= 32): the outputs of both (logits, topk_idx,
// topk_w, counts, offsets, row_of_copy, copy_of_row, x_perm).  ws_words:
// route_permute_hist_words(n_tok, n_exp) int32 of scratch, 128-byte aligned
// and zero before the first launch: the grid barrier's words (the kernel
// leaves them ready for the next launch) and the per-tile expert
// histograms.  D must be a multiple of 32.
int64_t route_permute_hist_words(int n_tok, int n_exp);
cudaError_t launch_route_permute(const RouteShape& s, int d, const void* x, const void* w_gate, const float* bias,
                                 float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                 int32_t* row_of_copy, int32_t* copy_of_row, void* x_perm, int32_t* ws_words,
                                 int32_t* status, cudaStream_t st);
// The router's tail in one launch (E <= 1024): the logits as the ordered fp32
// sum of their ks contraction slices (1 <= ks <= 4; part: [ks][N][E]; ks ==
// 1: part is the logits, not rewritten), per-token top-K over fp32 keys (logits + bias),
// weights renormalised from the unbiased logits, the expert histogram
// (counts) and its exclusive scan (offsets[0] = 0, offsets[e+1] =
// offsets[e] + counts[e]; a total other than N*K sets DEV_BAD_OFFSETS).
// acc: E int32 and ticket: one int32, zero before the launch (the kernel
// leaves them zero).
cudaError_t launch_topk_scan(const RouteShape& s, const float* part, int ks, float* logits, const float* bias,
                             int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* acc,
                             int32_t* ticket, int32_t* status, cudaStream_t st);
// Route-bias update from the histogram (mode 0: listing form, 1: +-gamma).
cudaError_t launch_update_bias(const int32_t* counts, int n_exp, float* bias, float gamma, int mode,
                               cudaStream_t st);

// The stable expert-major permutation maps.  Up to 65536 copies run in one
// CTA with no scratch (unless `chunked`); otherwise, or with `chunked`, the
// token-chunked form runs with block_counts/block_base as
// [num_chunks(n_tok), n_exp] int32 scratch.  Both give the same maps.
int permute_num_chunks(int n_tok);
cudaError_t launch_permute_maps(int n_tok, int n_exp, int top_k, const int32_t* topk_idx, const int32_t* offsets,
                                int32_t* block_counts, int32_t* block_base, int32_t* row_of_copy,
                                int32_t* copy_of_row, int32_t* status, cudaStream_t st, bool chunked = false);
// moe_permute in one launch (maps and rows; decoupled look-back over
// 16-token chunks).  look: permute_single_pass_look_words() uint64 and ctl:
// three int32 (chunk ticket, done counter, generation), all zero after
// moe_workspace_init; the kernel leaves ctl ready for the next call.
int64_t permute_single_pass_look_words(int n_tok, int n_exp);
cudaError_t launch_permute_single_pass(int n_tok, int n_exp, int top_k, int d, const int32_t* topk_idx,
                                       const int32_t* offsets, const void* x, int32_t* row_of_copy,
                                       int32_t* copy_of_row, void* x_perm, unsigned long long* look, int32_t* ctl,
                                       int32_t* status, cudaStream_t st);
// The same with the rows quantised to MXFP8 on the way (each token row read
// and quantised once, as launch_mx_quant_rows does): codes [R, d] and scales
// [d/32][ld] of the permuted rows; tok_codes / tok_scales (nullable): the
// token rows' codes [n_tok, d] and scales [d/32][tok_ld].  d % 32 == 0.
cudaError_t launch_permute_single_pass_mxfp8(int n_tok, int n_exp, int top_k, int d, const int32_t* topk_idx,
                                             const int32_t* offsets, const void* x, int32_t* row_of_copy,
                                             int32_t* copy_of_row, uint8_t* codes, uint8_t* scales, int64_t ld,
                                             uint8_t* tok_codes, uint8_t* tok_scales, int64_t tok_ld,
                                             unsigned long long* look, int32_t* ctl, int32_t* status,
                                             cudaStream_t st);
// x_perm[row_of_copy[t*K+k]] = x[t] (bf16 rows of d elements).
cudaError_t launch_permute_rows(int n_tok, int d, int top_k, const void* x, const int32_t* row_of_copy,
                                void* x_perm, cudaStream_t st);
// out[t] = sum_k g[t,k] * y_perm[row_of_copy[t*K+k]] (+ y_shared[t]), fp32 sum, bf16 store.
cudaError_t launch_combine(int n_tok, int d, int top_k, const void* y_perm, const int32_t* row_of_copy,
                           const float* topk_w, const void* y_shared, void* out, cudaStream_t st);
// dYw[row] = bf16(g * dY[t]); dg[t,k] = <dY[t], y_perm[row]>; dl[t,k] = router logit gradient.
// With q_codes, also the MXFP8 codes [R, D] of the bf16 dYw rows along D and
// their scale bytes q_scales[(col / 32) * q_ld + row] (the row-wise layout of
// launch_mx_quant_rows with one group).
cudaError_t launch_combine_bwd(int n_tok, int d, int top_k, int gate, const void* dy, const void* y_perm,
                               const int32_t* row_of_copy, const float* topk_w, const float* logits, int n_exp,
                               const int32_t* topk_idx, void* dyw, float* dg, float* dl, cudaStream_t st,
                               uint8_t* q_codes = nullptr, uint8_t* q_scales = nullptr, int64_t q_ld = 0);
// dW_g[e] = sum over the rows r of expert e of dl[copy_of_row[r]] * x_perm[r] (fp32).
// x_rows is x_perm [R,D] (gather_k = 0) or x [N,D] read in permuted order,
// row r = x[copy_of_row[r] / gather_k] (gather_k = top_k).
// Scratch (in floats) of launch_dwgate: 64-row chunk partials and the chunk prefix.
size_t dwgate_partial_floats(int n_tok, int top_k, int n_exp, int d);
cudaError_t launch_dwgate(int n_tok, int top_k, int n_exp, int d, const int32_t* offsets, const int32_t* copy_of_row,
                          const float* dl, const void* x_rows, int gather_k, float* scratch, float* dw_gate,
                          cudaStream_t st);
// Capacity (drop) mode: from the dropless permutation (offsets, row_full),
// keep at most `cap` copies per expert (the first in token order) in a
// compact expert-major layout: kept_offsets [E+1], row_of_copy [R] (-1 for a
// dropped copy), copy_of_row for the kept rows, n_dropped (nullable).
cudaError_t launch_capacity_maps(int n_tok, int n_exp, int top_k, const int32_t* topk_idx, const int32_t* offsets,
                                 const int32_t* row_full, int cap, int32_t* kept_offsets, int32_t* row_of_copy,
                                 int32_t* copy_of_row, int32_t* n_dropped, cudaStream_t st);
// dx[t] = sum_k dx_perm[row(t,k)] + sum_k dl[t,k] * W_g[idx[t,k]] (+ dx_shared[t]); bf16 out.
cudaError_t launch_unpermute_dx(int n_tok, int d, int top_k, const void* dx_perm, const int32_t* row_of_copy,
                                const float* dl, const int32_t* topk_idx, const void* w_gate,
                                const void* dx_shared, void* dx, cudaStream_t st);
// dst[0] = 0, dst[1] = n (device offsets of a single dense group).
cudaError_t launch_dense_offsets(int32_t* dst, int n, cudaStream_t st);

}  // namespace moe
