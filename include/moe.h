/*
 * moe.h - C ABI of libmoe, a single-GPU dropless Mixture-of-Experts layer
 * (forward and backward) written as hand-made CUDA kernels for sm_103a.
 *
 * What the layer computes is the single-device MoE layer of "LLM
 * Infrastructure Engineering 08: MoE Training Engineering" (quant67):
 *   §4.1 / §4.3  router: logits = x W_g^T (fp32, §12.7); top-K selection;
 *                softmax (then renormalised over the K selected) or sigmoid
 *                of the selected logits renormalised to sum 1;
 *   §6.3         DeepSeek-V3 bias-adjusted selection: top-K ranks
 *                logits + route_bias, weights use the unbiased logits;
 *   §9           SwiGLU experts y = w2(silu(w1 x) * w3 x) (no bias), every
 *                token copy computed (dropless: no capacity, no drop, no pad,
 *                "Accelerating Dropless MoE Training in JAX with NVIDIA
 *                Transformer Engine" ¶2-¶3), results weighted and summed back
 *                per token; shared expert added to every token (§5 formula);
 *                load statistics and update_balance_bias;
 *   §12.5        dispatch as a sort of token copies by destination, combine
 *                as unsort + weighted sum over K.
 * The backward is the exact derivative of that forward (§11.3: experts that
 * received no token get zero weight gradient; the route bias gets none).
 *
 * Conventions (all entry points):
 *  - Every pointer is device memory owned by the caller unless stated; the
 *    library allocates nothing and frees nothing.  bf16 buffers are passed as
 *    void* and hold IEEE bfloat16 values, row-major.
 *  - Notation: N = n_tok, D = d_model, F = d_ff, E = n_exp, K = top_k,
 *    R = N*K rows of the permuted (expert-major) buffers, Fs = d_ff_shared.
 *  - Weights use the nn.Linear layout: W_g [E,D]; w1, w3 [E,F,D];
 *    w2 [E,D,F]; shared ws1, ws3 [Fs,D], ws2 [D,Fs].
 *  - Buffers must be 16-byte aligned; D, F and Fs must be multiples of 64;
 *    1 <= K <= min(E, 32); E <= 1024; R < 2^31.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work: no host synchronisation and no host read of device data,
 *    so a sequence of calls can be captured in a CUDA graph.
 *  - Errors the host can detect (bad sizes, null or misaligned pointers,
 *    workspace too small) return a status before anything is enqueued.
 *    Errors found on the device (an expert index out of range, a bounded
 *    wait that timed out) set bits in the status word at the start of the
 *    workspace; read it with moe_get_device_status.
 *  - Workspace: `ws` must hold moe_workspace_size() bytes and be cleared once
 *    with moe_workspace_init.  One workspace must not be used by two calls
 *    that may run concurrently.
 */
#ifndef RAGGED_GROUPED_GEMM_GB300_MOE_H
#define RAGGED_GROUPED_GEMM_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, size out of range */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE = 5        /* device status word reports an error */
} moe_status_t;

/* Device status bits (moe_get_device_status). */
#define MOE_DEV_TIMEOUT 1      /* a bounded wait inside a kernel ran out */
#define MOE_DEV_BAD_INDEX 2    /* an expert index outside [0, E) */
#define MOE_DEV_BAD_OFFSETS 4  /* the histogram did not sum to N*K, or (permute)
                                  offsets inconsistent with the expert indices */

/* Layer description; the pages' MoELayer(d_model, d_ff, n_experts, top_k,
 * n_shared, use_bias_balance) constructor (§9). */
typedef struct {
  int32_t n_tok;       /* N: tokens in the batch (B*T) */
  int32_t d_model;     /* D */
  int32_t d_ff;        /* F: routed expert hidden size */
  int32_t n_exp;       /* E: routed experts */
  int32_t top_k;       /* K */
  int32_t gate;        /* 0: softmax top-K renorm (§4.1); 1: sigmoid renorm (§4.3) */
  int32_t use_bias;    /* 1: select on logits + route_bias (§6.3) */
  int32_t n_shared;    /* 0 or 1 shared expert (§5) */
  int32_t d_ff_shared; /* Fs */
  int32_t precision;   /* 0: bf16; 1: MXFP8 expert GEMM operands; 2: FP8 weights (bf16 activations); fp32 accumulation */
} moe_desc_t;

/* Expert weights (all bf16, nn.Linear layout, see above).  ws1/ws3/ws2 are
 * ignored when n_shared == 0. */
typedef struct {
  const void* w1;
  const void* w3;
  const void* w2;
  const void* ws1;
  const void* ws3;
  const void* ws2;
} moe_expert_weights_t;

/* Activations the forward writes for the backward (bf16).  a1 = x_e w1_e^T,
 * a3 = x_e w3_e^T, h = silu(a1) * a3, per permuted row [R,F]; the shared
 * expert's a1s, a3s, hs are [N,Fs].  a1/a3/a1s/a3s may be NULL for an
 * inference-only forward; h (and hs with a shared expert) are required. */
typedef struct {
  void* a1;
  void* a3;
  void* h;
  void* a1s;
  void* a3s;
  void* hs;
} moe_ffn_saved_t;

/* Everything the backward reads from the forward (all written by the
 * forward entry points, see each). */
typedef struct {
  const void* x;               /* [N,D] bf16 layer input */
  const void* x_perm;          /* [R,D] bf16 from moe_permute */
  const float* logits;         /* [N,E] fp32 from moe_route */
  const int32_t* topk_idx;     /* [N,K] */
  const float* topk_w;         /* [N,K] */
  const int32_t* offsets;      /* [E+1] */
  const int32_t* row_of_copy;  /* [R] */
  const int32_t* copy_of_row;  /* [R] */
  const void* a1;              /* [R,F] */
  const void* a3;              /* [R,F] */
  const void* h;               /* [R,F] */
  const void* y_perm;          /* [R,D] from moe_grouped_ffn */
  const void* a1s;             /* [N,Fs] */
  const void* a3s;             /* [N,Fs] */
  const void* hs;              /* [N,Fs] */
  /* Capacity (drop) mode only, NULL otherwise: the dropless offsets [E+1]
   * from moe_route and copy_of_row [R] from moe_permute_capacity.  The
   * router weight gradient sums over every copy, dropped or kept. */
  const int32_t* offsets_full;
  const int32_t* copy_of_row_full;
} moe_fwd_state_t;

/* Gradients written by moe_backward (fp32 unless stated).  dg and dlogits
 * may be NULL; the shared gradients are ignored when n_shared == 0. */
typedef struct {
  void* dx;          /* [N,D] bf16: input gradient (experts + router) */
  float* dw_gate;    /* [E,D] */
  float* dw1;        /* [E,F,D] (zero for experts with no token) */
  float* dw3;        /* [E,F,D] */
  float* dw2;        /* [E,D,F] */
  float* dws1;       /* [Fs,D] */
  float* dws3;       /* [Fs,D] */
  float* dws2;       /* [D,Fs] */
  float* dg;         /* [N,K] d loss / d topk_w */
  float* dlogits;    /* [N,K] d loss / d logits at the selected experts (0 elsewhere) */
} moe_grads_t;

/* Library and ABI identification. */
MOE_API int32_t moe_abi_version(void);
MOE_API const char* moe_status_string(moe_status_t s);

/* Bytes of workspace the forward calls (route, permute, grouped_ffn,
 * combine) and the backward call need for `d`.  fwd_bytes <= bwd_bytes; a
 * workspace of bwd_bytes serves every call.  Either output may be NULL. */
MOE_API moe_status_t moe_workspace_size(const moe_desc_t* d, size_t* fwd_bytes, size_t* bwd_bytes);

/* Clear the whole workspace (ws_bytes, enqueued on stream): the device
 * status words and the counters and look-back words the router and the
 * permutation keep there start at zero (every call leaves them ready for
 * the next one).  Once per workspace, before its first use. */
MOE_API moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then copy the two device status words (bits, site)
 * to `status_host[0..1]`.  The only call that blocks the host. */
MOE_API moe_status_t moe_get_device_status(const void* ws, int32_t* status_host, void* stream);

/* Router (§4.1, §4.3, §6.3, §9 step 1) and expert histogram (§9 step 4,
 * §12.5 bincount):
 *   logits[N,E] (fp32 out) = x[N,D] (bf16) * w_gate[E,D]^T  (tensor cores,
 *                            fp32 accumulation, deterministic.  E <= 32: the
 *                            whole router is one kernel (warp-level MMA over
 *                            16-token tiles, the contraction cut into 16
 *                            slices added in slice order, then the selection
 *                            and histogram below).  E > 32: the grouped GEMM
 *                            on 128-token tiles; with few tiles the
 *                            contraction runs in up to 4 slices whose fp32
 *                            partial products, kept in the workspace, are
 *                            added in slice order by one more kernel that
 *                            also does the selection, histogram and scan);
 *   topk_idx[N,K] (out)    = the K experts with the largest
 *                            logits + bias (bias [E] fp32, NULL when the layer
 *                            has none), sorted by rank; equal keys: lower
 *                            expert index first; -0.0 == +0.0; NaN lowest;
 *   topk_w[N,K] (fp32 out) = renormalised gate weights (softmax over all E
 *                            then p_sel/sum p_sel, or sigmoid(l_sel)/sum);
 *   counts[E] (int32 out)  = copies routed to each expert;
 *   offsets[E+1] (out)     = exclusive prefix sum of counts.
 * Needs the forward workspace. */
MOE_API moe_status_t moe_route(const moe_desc_t* d, const void* x, const void* w_gate, const float* bias,
                       float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                       void* ws, size_t ws_bytes, void* stream);

/* The same selection, weights, histogram and offsets from given fp32
 * logits [N,E] (input).  Used when logits come from elsewhere. */
MOE_API moe_status_t moe_route_from_logits(const moe_desc_t* d, const float* logits, const float* bias,
                                   int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                   void* ws, size_t ws_bytes, void* stream);

/* Router and dispatch together (§4.1, §4.3, §9 steps 1-4, §12.5 sort by
 * destination): moe_route followed by moe_permute on the same tokens, in one
 * launch, for E <= 32 and bf16 rows (precision 0 or 2).  The outputs of both
 * calls, bit-identical to them (logits, topk_idx, topk_w, counts, offsets as
 * moe_route; row_of_copy, copy_of_row, x_perm as moe_permute).  A
 * cooperative launch: each CTA routes its tiles (at most 16 tokens each, as
 * many per CTA as the batch allows) and publishes their expert histograms, a grid-wide barrier follows (bounded: a
 * wait that runs out sets MOE_DEV_TIMEOUT, site 710), then each CTA finds its
 * tiles' first rows from the histograms and copies its token rows while they
 * are still in L2.  Needs the forward workspace (its per-tile histograms are
 * part of it).  Errors: MOE_ERR_INVALID_ARG for E > 32, precision 1 (use
 * moe_permute_mxfp8), unaligned or missing pointers; the launch's own error
 * otherwise (for instance when the GPU cannot run a cooperative launch). */
MOE_API moe_status_t moe_route_permute(const moe_desc_t* d, const void* x, const void* w_gate, const float* bias,
                                       float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                       int32_t* offsets, int32_t* row_of_copy, int32_t* copy_of_row, void* x_perm,
                                       void* ws, size_t ws_bytes, void* stream);

/* Dispatch (§12.5 sort by destination; §9 mask/nonzero order): a stable
 * counting sort of the copies c = t*K+k by expert, ascending token inside
 * an expert.  row_of_copy[c] (out) is the permuted row of copy c;
 * copy_of_row[r] (out) its inverse; x_perm[r,:] (out, bf16 [R,D]) =
 * x[copy_of_row[r]/K,:].  Rows of expert e are offsets[e]..offsets[e+1]-1.
 * `offsets` comes from moe_route.  One launch: each 16-token chunk finds its
 * first row per expert from the preceding chunks' published counts (bounded
 * waits; MOE_DEV_TIMEOUT if one ran out) and copies its rows.  A copy whose
 * row would fall outside its expert's rows or [0, R) gets row -1
 * (MOE_DEV_BAD_OFFSETS); an expert index outside [0, E) gets row -1
 * (MOE_DEV_BAD_INDEX).  Needs the forward workspace. */
MOE_API moe_status_t moe_permute(const moe_desc_t* d, const void* x, const int32_t* topk_idx, const int32_t* offsets,
                         int32_t* row_of_copy, int32_t* copy_of_row, void* x_perm, void* ws, size_t ws_bytes,
                         void* stream);

/* The maps of moe_permute alone (row_of_copy, copy_of_row; no row is
 * copied), for moe_grouped_ffn_gather.  Same arguments, results and errors
 * as moe_permute without x and x_perm.  Needs the forward workspace. */
MOE_API moe_status_t moe_permute_maps(const moe_desc_t* d, const int32_t* topk_idx, const int32_t* offsets,
                                      int32_t* row_of_copy, int32_t* copy_of_row, void* ws, size_t ws_bytes,
                                      void* stream);

/* Ragged grouped SwiGLU FFN (§9 Expert; grouped GEMM of "Accelerating
 * Dropless MoE Training in JAX with NVIDIA Transformer Engine" ¶5): for every
 * expert e and its rows r in [offsets[e], offsets[e+1]):
 *   a1 = x_perm[r] w1_e^T, a3 = x_perm[r] w3_e^T, h[r] = silu(a1) * a3,
 *   y_perm[r] = h[r] w2_e^T  (bf16 out [R,D], unweighted).
 * Both GEMMs run as one persistent tcgen05 launch each over all experts,
 * reading the group sizes from `offsets` on the device.  With a shared
 * expert the same FFN of ws1/ws3/ws2 runs over x (all N tokens) into
 * y_shared [N,D] (bf16 out); y_shared is ignored otherwise.  `saved`
 * receives the activations (see moe_ffn_saved_t). */
MOE_API moe_status_t moe_grouped_ffn(const moe_desc_t* d, const void* x_perm, const int32_t* offsets, const void* x,
                             const moe_expert_weights_t* w, const moe_ffn_saved_t* saved, void* y_perm,
                             void* y_shared, void* ws, size_t ws_bytes, void* stream);

/* moe_grouped_ffn with the dispatch fused into GEMM1's operand loads
 * ("LLM Infrastructure Engineering 08: MoE Training Engineering" §9
 * engineering notes: scatter + grouped GEMM): GEMM1 reads the rows of
 * expert e straight from the token matrix x [N,D] (bf16), row r being token
 * copy_of_row[r] / K, by TMA four-row gathers, so no permuted copy of the
 * tokens is written or read.  copy_of_row and offsets come from
 * moe_permute_maps (or moe_permute); every other argument, output and saved
 * activation as moe_grouped_ffn, with bit-identical results.  bf16 layers
 * only (MOE_ERR_UNSUPPORTED otherwise).  A training step still needs
 * x_perm for the w1/w3 weight gradients (moe_permute). */
MOE_API moe_status_t moe_grouped_ffn_gather(const moe_desc_t* d, const void* x, const int32_t* copy_of_row,
                                            const int32_t* offsets, const moe_expert_weights_t* w,
                                            const moe_ffn_saved_t* saved, void* y_perm, void* y_shared, void* ws,
                                            size_t ws_bytes, void* stream);

/* Combine (§9 index_add_ of weighted outputs plus shared expert; §12.5
 * unsort + K-sum): out[t] = sum_{k<K} topk_w[t,k] * y_perm[row_of_copy[t*K+k]]
 * + y_shared[t] (y_shared NULL: no shared term), summed in fp32 in rank
 * order, stored bf16 [N,D].  A token-major gather, so deterministic. */
MOE_API moe_status_t moe_combine(const moe_desc_t* d, const void* y_perm, const int32_t* row_of_copy, const float* topk_w,
                         const void* y_shared, void* out, void* stream);

/* Backward of the layer for the upstream gradient dy [N,D] (bf16 input):
 * combine backward (dYw = g*dY per permuted row, dg = <dY, y_perm>), grouped
 * data-gradient GEMM through w2 with the SwiGLU derivative fused in its
 * epilogue, grouped data-gradient GEMM through w1|w3, grouped weight-gradient
 * GEMMs (contraction over each expert's ragged rows, fp32 out, zero for
 * empty experts), the shared expert's backward, the router logit gradient
 * (softmax-renorm: g_k (dg_k - sum_j g_j dg_j); sigmoid-renorm:
 * s_k (1-s_k)/S (dg_k - sum_j g_j dg_j); no gradient to route_bias), the
 * router weight gradient dw_gate = dlogits^T x and the input gradient
 * dx = sum_k dx_perm + dlogits W_g (+ shared).  Needs the backward workspace. */
MOE_API moe_status_t moe_backward(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_t* w,
                          const moe_fwd_state_t* st, const void* dy, const moe_grads_t* g, void* ws,
                          size_t ws_bytes, void* stream);

/* Online route-bias update (§9 update_balance_bias, §6.3), in place on
 * bias[E] (fp32) from counts[E] of the last batch, load_stat = counts/sum:
 *   mode 0 (listing): bias -= gamma * sign(load_stat - 1/E) * max(load_stat, 1e-6)
 *   mode 1 (prose):   bias -= gamma * sign(load_stat - 1/E)
 * in fp32 with every operation rounded separately.  An empty batch leaves
 * the bias unchanged. */
MOE_API moe_status_t moe_update_bias(const moe_desc_t* d, const int32_t* counts, float* bias, float gamma, int32_t mode,
                             void* stream);

/* Capacity-factor mode (§6.4 "Capacity Factor and Token Drop", §2.2 GShard):
 * the comparison case of the dropless layer.  capacity = ceil(capacity_factor
 * * (N / E * K)) copies per expert; each expert keeps its first copies in
 * token order and drops the rest, which contribute nothing to the combine
 * (the token keeps only its residual path, outside the layer); the kept gate
 * weights are not renormalised.
 * Inputs: x [N,D], topk_idx [N,K], offsets [E+1] (dropless, from moe_route).
 * Outputs: row_of_copy_full [R], copy_of_row_full [R] (the dropless maps of
 * moe_permute), kept_offsets [E+1], row_of_copy [R] (-1 for a dropped copy),
 * copy_of_row (first kept_offsets[E] entries), x_perm [R,D] (first
 * kept_offsets[E] rows), n_dropped [1] (device int32, nullable).  The expert
 * GEMMs, combine and backward then run on kept_offsets / row_of_copy /
 * copy_of_row / x_perm unchanged (moe_fwd_state_t.offsets_full and
 * copy_of_row_full take the dropless maps).  bf16 only (d->precision 0).
 * Needs the forward workspace. */
MOE_API moe_status_t moe_permute_capacity(const moe_desc_t* d, const void* x, const int32_t* topk_idx,
                                          const int32_t* offsets, double capacity_factor,
                                          int32_t* row_of_copy_full, int32_t* copy_of_row_full,
                                          int32_t* kept_offsets, int32_t* row_of_copy, int32_t* copy_of_row,
                                          void* x_perm, int32_t* n_dropped, void* ws, size_t ws_bytes,
                                          void* stream);

/* Auxiliary load-balancing loss (§6.2, GShard form) of the routing that
 * produced `logits` [N,E] (fp32, from moe_route) and `counts` [E]:
 *   loss[0] = coef * E * sum_i f_i P_i,  f_i = counts_i / N (mean of the
 *   top-K mask), P_i = mean over tokens of the softmax over all E logits
 *   (softmax gate) or of the sigmoid scores normalised over all E (sigmoid
 *   gate; the pages give no P for it).
 * dlogits_aux [N,E] (fp32, NULL: not computed) receives d loss / d logits with
 * f held fixed (the selection is discrete); the caller adds it to the
 * router's logit gradient.  Deterministic (fixed-order sums).  loss is a
 * device pointer.  Needs the forward workspace. */
MOE_API moe_status_t moe_aux_loss(const moe_desc_t* d, const float* logits, const int32_t* counts, float coef,
                                  float* loss, float* dlogits_aux, void* ws, size_t ws_bytes, void* stream);

/* Load monitor statistics (§13.9) over a window of routing histograms:
 * counts_hist [n_hist, n_exp] int32 on the device, one row per step (e.g. the
 * counts of the last 100 steps; rows must not sum to 0).  Each row becomes
 * the load fraction counts / sum (fp32); the window mean r (fp64) gives
 *   stats[0] = min_e r_e, stats[1] = -sum_e r_e log(r_e + 1e-9),
 *   stats[2] = number of experts with r_e < 0.3 / n_exp (as a float).
 * stats is a device pointer to 3 floats.  n_exp <= 1024. */
MOE_API moe_status_t moe_monitor_stats(int32_t n_exp, const int32_t* counts_hist, int32_t n_hist, float* stats,
                                       void* stream);

/* ---------------------------------------------------------------- MXFP8 --
 * The MXFP8 forward path: the expert GEMMs read their operands as MXFP8 (OCP
 * Microscaling v1.0: E4M3 elements, one E8M0 power-of-two scale per 32
 * consecutive elements along the contraction dimension), halving the bytes of
 * weights and activations ("Accelerating Dropless MoE Training in JAX with
 * NVIDIA Transformer Engine" ¶6: group-aware MXFP8 grouped GEMM; "LLM
 * Infrastructure Engineering 08: MoE Training Engineering" §13.6: fine-
 * grained scaling, fp32 accumulation).  Block scale 2^(floor(log2 amax) - 8);
 * elements rounded to nearest even and saturated at +-448; an all-zero block
 * has scale byte 0.  Scales are stored k-block-major: for a matrix [rows,
 * cols] (cols = contraction dimension) the byte of row r, block b is at
 * scales[b * scale_ld + r] with scale_ld >= rows and a multiple of 16.
 * The tensor cores run block-scaled MMAs (tcgen05 kind::mxf8f6f4 with the
 * E8M0 scales in tensor memory) with fp32 accumulation.  The backward is
 * moe_backward_mxfp8 (every expert GEMM with MXFP8 operands) or moe_backward
 * (bf16) on the bf16 activations the MXFP8 forward saved. */

/* Round up to the scale leading dimension the library expects (multiple of 16). */
#define MOE_MX_SCALE_LD(rows) ((((rows) + 15) / 16) * 16)

/* MXFP8 expert weights: codes (uint8) in the weights' layouts, scales
 * [groups][K/32][N] per matrix [N,K] (K = contraction dimension):
 *   w1, w3 codes [E,F,D], scales [E, D/32, F];  w2 codes [E,D,F], scales [E, F/32, D];
 *   ws1, ws3 codes [Fs,D], scales [D/32, Fs];   ws2 codes [D,Fs], scales [Fs/32, D]. */
typedef struct {
  const void* w1;
  const void* w1_scale;
  const void* w3;
  const void* w3_scale;
  const void* w2;
  const void* w2_scale;
  const void* ws1;
  const void* ws1_scale;
  const void* ws3;
  const void* ws3_scale;
  const void* ws2;
  const void* ws2_scale;
} moe_expert_weights_mx_t;

/* Quantise bf16 src [groups, rows, cols] rowwise to MXFP8 along cols: codes
 * [groups, rows, cols] and scales [groups, cols/32, scale_ld].  cols must be
 * a multiple of 32; scale_ld >= rows and a multiple of 16.  Used for weights
 * (once per optimiser step, outside the layer). */
MOE_API moe_status_t moe_quantize_mxfp8(const void* src, int64_t groups, int64_t rows, int64_t cols, void* codes,
                                        void* scales, int64_t scale_ld, void* stream);

/* Quantise bf16 src [groups, rows, cols] to MXFP8 along ROWS and store it
 * transposed: codes [groups, cols, rows] and scales [groups, rows/32,
 * scale_ld] (scale_ld >= cols, a multiple of 16; rows a multiple of 32).  The
 * weights' copies for the backward's data-gradient GEMMs, whose contraction
 * runs over the other weight dimension: w2 [E,D,F] -> codes [E,F,D] with
 * scales [E,D/32,F]; w1, w3 [E,F,D] -> codes [E,D,F] with scales [E,F/32,D]
 * (once per optimiser step, outside the layer). */
MOE_API moe_status_t moe_quantize_mxfp8_t(const void* src, int64_t groups, int64_t rows, int64_t cols, void* codes,
                                          void* scales, int64_t scale_ld, void* stream);

/* moe_permute with MXFP8 quantisation fused in: the same row_of_copy /
 * copy_of_row maps, and the permuted rows as codes xq_perm [R,D] with scales
 * xs_perm [D/32, MOE_MX_SCALE_LD(R)]; optionally (xq_tok non-NULL) the
 * token-order rows xq_tok [N,D], xs_tok [D/32, MOE_MX_SCALE_LD(N)] for the
 * shared expert.  d->precision must be 1.  Needs the forward workspace.
 * Where moe_permute runs in one launch (ceil(N/16) * E <= 131072), so does
 * this: each token row is read and quantised once, and its codes and scale
 * bytes are written to its K rows (and its token row); the codes are those
 * of moe_quantize_mxfp8 applied to the permuted rows. */
MOE_API moe_status_t moe_permute_mxfp8(const moe_desc_t* d, const void* x, const int32_t* topk_idx,
                                       const int32_t* offsets, int32_t* row_of_copy, int32_t* copy_of_row,
                                       void* xq_perm, void* xs_perm, void* xq_tok, void* xs_tok, void* ws,
                                       size_t ws_bytes, void* stream);

/* moe_grouped_ffn with MXFP8 operands: GEMM1 reads xq_perm/xs_perm and the
 * MXFP8 w1, w3; its epilogue computes h = silu(a1) * a3 and quantises it to
 * MXFP8 along F (kept in the workspace); GEMM2 reads it with w2 and writes
 * y_perm [R,D] bf16.  The shared expert does the same from xq_tok/xs_tok into
 * y_shared.  `saved` may hold bf16 a1, a3, h (and a1s, a3s, hs) for a bf16
 * backward, or NULL pointers.  d->precision must be 1. */
MOE_API moe_status_t moe_grouped_ffn_mxfp8(const moe_desc_t* d, const void* xq_perm, const void* xs_perm,
                                           const int32_t* offsets, const void* xq_tok, const void* xs_tok,
                                           const moe_expert_weights_mx_t* w, const moe_ffn_saved_t* saved,
                                           void* y_perm, void* y_shared, void* ws, size_t ws_bytes, void* stream);

/* Backward of the MXFP8 layer: the steps of moe_backward with every expert
 * GEMM on MXFP8 operands, each quantised along that GEMM's contraction
 * ("Accelerating Dropless MoE Training in JAX with NVIDIA Transformer Engine"
 * ¶6, group-aware MXFP8 grouped GEMM, read for the backward):
 *   dh = dYw w2      : dYw quantised along D, w2 along D (wt->w2: codes
 *                      [E,F,D], scales [E,D/32,F] from moe_quantize_mxfp8_t),
 *                      SwiGLU derivative in the epilogue -> da1, da3 (bf16);
 *   dx = da1 w1 + da3 w3 : da1, da3 quantised along F, w1, w3 along F
 *                      (wt->w1, wt->w3: codes [E,D,F], scales [E,F/32,D]);
 *   dW2 = dYw^T h, dW1 = da1^T x, dW3 = da3^T x : operands quantised along
 *                      each expert's tokens, blocks restarting at the
 *                      expert's first row (fp32 out, zero for empty experts).
 * The shared expert is the same with one group (wt->ws1/ws3: codes [D,Fs],
 * scales [Fs/32,D]; wt->ws2: codes [Fs,D], scales [D/32,Fs]).  The combine
 * and router backward are those of moe_backward.  s->x_perm is not read (the
 * permuted input is gathered from s->x); s->a1, a3, h (a1s, a3s, hs) are the
 * bf16 activations saved by moe_grouped_ffn_mxfp8.  d->precision must be 1;
 * needs the backward workspace of that description. */
MOE_API moe_status_t moe_backward_mxfp8(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_mx_t* wt,
                                        const moe_fwd_state_t* s, const void* dy, const moe_grads_t* g, void* ws,
                                        size_t ws_bytes, void* stream);

/* ------------------------------------------------------- FP8 weights --
 * The FP8 training recipe of "LLM Infrastructure Engineering 08: MoE
 * Training Engineering" §13.6: forward act(BF16) x weight(FP8) -> BF16,
 * backward grad(BF16) x weight_T(FP8) -> BF16, per-tile scaling, FP32
 * accumulation.  Weights are E4M3 codes with one fp32 scale per 128 x 128
 * tile (scale = tile amax / 448, reading of "per-tile"); one tile grid serves
 * both the forward and the transposed (data-gradient) use.  The GEMMs
 * dequantise each weight tile to bf16 in shared memory (code x scale, the
 * fp32 product rounded to bf16) and run bf16 tensor-core MMAs; activations
 * stay bf16 and the weight gradients are bf16 GEMMs with fp32 output, as in
 * moe_backward.  d->precision must be 2. */

/* Quantise bf16 weights src [groups, rows, cols] per 128 x 128 tile: codes
 * [groups, rows, cols] (uint8 E4M3, w / scale rounded to nearest even,
 * saturating at 448) and scales [groups, ceil(rows/128), ceil(cols/128)]
 * (fp32).  cols must be a multiple of 16.  Once per optimiser step. */
MOE_API moe_status_t moe_quantize_fp8_tile(const void* src, int64_t groups, int64_t rows, int64_t cols,
                                           void* codes, float* scales, void* stream);

/* moe_grouped_ffn with FP8 weights: the moe_expert_weights_mx_t fields hold
 * the codes (w1, w3 [E,F,D]; w2 [E,D,F]; ws1, ws3 [Fs,D]; ws2 [D,Fs]) and, in
 * the *_scale fields, the fp32 tile scales from moe_quantize_fp8_tile.  Other
 * arguments, outputs and saved activations as moe_grouped_ffn. */
MOE_API moe_status_t moe_grouped_ffn_fp8w(const moe_desc_t* d, const void* x_perm, const int32_t* offsets,
                                          const void* x, const moe_expert_weights_mx_t* wq,
                                          const moe_ffn_saved_t* saved, void* y_perm, void* y_shared, void* ws,
                                          size_t ws_bytes, void* stream);

/* moe_backward of the FP8-weight layer: the data gradients through w2 and
 * w1|w3 read the same codes and tile scales as moe_grouped_ffn_fp8w; the
 * rest as moe_backward. */
MOE_API moe_status_t moe_backward_fp8w(const moe_desc_t* d, const void* w_gate, const moe_expert_weights_mx_t* wq,
                                       const moe_fwd_state_t* s, const void* dy, const moe_grads_t* g, void* ws,
                                       size_t ws_bytes, void* stream);

/* moe_permute without a workspace (no counterpart in the pages; an addition
 * of this library for callers that cannot allocate).  Same inputs, outputs
 * and results as moe_permute, for callers that cannot give the library any
 * device memory of its own: for example a plugin that its host application
 * calls with nothing but input and output buffers and no allocator, or a
 * loop running under a fixed memory budget reserved up front, where a new
 * allocation is not allowed (cudaMalloc may block and synchronise the GPU).
 * The per-chunk tables moe_permute keeps in the workspace live here in one
 * fixed 512 KiB device array inside the library, resident on every GPU that
 * loads it until the process exits.  Limit: ceil(n_tok/128) * n_exp must not
 * exceed 65536; larger sizes return MOE_ERR_WORKSPACE before anything is
 * enqueued.  The call allocates nothing.  Every call looks up the array's
 * device address on the current device (a host-side query, no device work),
 * so the address stays valid after a device reset; the first lookup on a
 * device may load the library's device code there, so make the first call
 * on each device before any stream capture.  All calls share the
 * one array (it keeps the last call's contents; every call rewrites the
 * parts it reads): calls whose work may overlap on the GPU race with each
 * other and must be serialised, e.g. issued on one stream.  Expert indices
 * outside [0, E) are skipped without a device status report (there is no
 * workspace to hold one). */
MOE_API moe_status_t moe_permute_noalloc(const moe_desc_t* d, const void* x, const int32_t* topk_idx,
                                         const int32_t* offsets, int32_t* row_of_copy, int32_t* copy_of_row,
                                         void* x_perm, void* stream);

/* Self-test of device failure detection (no counterpart in the pages; a
 * check of this library's own bounded waits).  Enqueues one small kernel
 * built from the wait routine every pipeline of the library uses, on
 * mbarriers that nothing ever arrives on: one wait has the limit `limit_ns`
 * (1 ns .. 1 s) and runs out, setting MOE_DEV_TIMEOUT in the status word at
 * the start of `ws` and `site` in the second word; a second wait with the
 * library's default limit (2 s) sees the first one's abort flag and returns
 * at once.  The kernel then exits normally, so the context stays usable.
 * `ws` needs at least 8 bytes (a layer workspace works); clear it with
 * moe_workspace_init first and read the result with moe_get_device_status. */
MOE_API moe_status_t moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, int32_t site,
                                               void* stream);

/* ---------------------------------------------------------- kernel timing --
 * Per-kernel timing of the grouped GEMMs (no counterpart in the pages; a
 * measurement aid of this library).  While enabled, every grouped-GEMM
 * launch of the entry points above is bracketed by two CUDA events recorded
 * on its stream, and its kind is noted:
 *   MOE_TIMING_GATE     router logits GEMM (moe_route);
 *   MOE_TIMING_FFN_FWD  expert GEMMs of the forward: GEMM1 (w1|w3 + SwiGLU)
 *                       and GEMM2 (w2), routed and shared, every precision;
 *   MOE_TIMING_DGRAD    data-gradient GEMMs of the backward (through w2 with
 *                       the SwiGLU derivative, through w1|w3);
 *   MOE_TIMING_WGRAD    weight-gradient GEMMs (dW1, dW3, dW2, routed and
 *                       shared).
 * The events are host driver objects (no device memory) that
 * moe_timing_enable creates, `capacity` pairs of them (1 .. 2^20), after
 * clearing earlier records; launches past the capacity, and launches on a
 * stream that is capturing a graph, are counted as untimed.  The recorded
 * events add two tiny commands per launch to the stream and nothing else.
 * moe_timing_read waits for the recorded events of `kind` (a host
 * synchronisation, unlike every other entry point) and returns the sum of
 * their elapsed times in milliseconds, the number of timed launches and
 * (nullable) the number of untimed ones since moe_timing_enable.
 * moe_timing_disable stops timing and destroys the events.  Process-wide
 * state; enable, read and disable must not race with launches from other
 * host threads. */
#define MOE_TIMING_GATE 0
#define MOE_TIMING_FFN_FWD 1
#define MOE_TIMING_DGRAD 2
#define MOE_TIMING_WGRAD 3
MOE_API moe_status_t moe_timing_enable(int32_t capacity);
MOE_API moe_status_t moe_timing_read(int32_t kind, double* total_ms, int64_t* launches, int64_t* untimed);
MOE_API moe_status_t moe_timing_disable(void);

#ifdef __cplusplus
}
#endif

#endif /* RAGGED_GROUPED_GEMM_GB300_MOE_H */
