"""Plain CPU oracle of the dropless MoE layer, forward and backward.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py``; never by the library.

Sources (page title, then section as numbered on that page):

* [MoE-Eng] "LLM Infrastructure Engineering 08: MoE Training Engineering"
  (quant67.com).  §4.1 softmax top-K gate listing; §4.3 sigmoid gate with
  top-K renormalisation; §5 shared + routed experts formula; §6.2 auxiliary
  load-balancing loss listing; §6.3 bias-adjusted selection; §9 "a simplified
  MoE layer" listing (SwiGLU ``Expert``, ``MoELayer.forward`` loop over experts,
  ``update_balance_bias``); §11.3 sparse backward; §12.5 EP skeleton
  (sort / bincount / unsort / K-sum); §12.7 fp32 gate; §13.9 monitor hook.
* [TE-JAX] "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer
  Engine" (technical analysis, ai.warp-studio.com), ¶2-¶3: dropless means
  every token copy is computed, with no capacity limit, no drop and no pad.

Precision.  The gate is computed in fp32 ([MoE-Eng] §12.7).  Routing
decisions (top-K keys, renormalised weights) are taken in fp32, the precision
the pages fix.  Expert arithmetic runs in ``dtype`` (fp32 by default, fp64 for
finite-difference pins).  Inputs are the bf16-valued buffers the GPU receives,
widened exactly.

Readings of points the pages leave open are stated where they are used:
tie-break (lower expert index wins), ranking the logits rather than the
softmax probabilities, -0.0 == +0.0 and NaN below every number, order of
copies inside an expert (ascending token), empty experts get zero weight
gradient, the bias update's window (the last batch) and its empty-batch case.
"""
from __future__ import annotations

import functools

import numpy as np

__all__ = [
    "gate_logits", "selection_keys", "topk_select", "topk_select_bruteforce",
    "gate_weights", "route", "histogram", "exclusive_offsets", "permutation",
    "swiglu_expert", "moe_forward", "moe_forward_dense_bruteforce",
    "moe_backward", "router_logit_grad", "update_bias", "aux_loss", "aux_loss_grad",
    "capacity", "permutation_capacity", "moe_forward_capacity",
    "monitor_stats", "load_stat",
]

F32 = np.float32


# ----------------------------------------------------------------------------
# Router ([MoE-Eng] §4.1, §4.3, §6.3, §9 steps 1)
# ----------------------------------------------------------------------------
def gate_logits(x: np.ndarray, w_gate: np.ndarray, dtype=F32) -> np.ndarray:
    """``logits = x W_g^T`` in fp32 ([MoE-Eng] §4.1 ``self.w_gate(x)``, §12.7 fp32 gate).

    x: [N, D], w_gate: [E, D] (nn.Linear weight layout).  Returns [N, E] in
    ``dtype`` (fp32, the pages' precision; fp64 only for finite-difference pins).
    """
    return np.matmul(x.astype(dtype), w_gate.astype(dtype).T).astype(dtype)


def selection_keys(logits: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """The values top-K ranks: ``logits + route_bias`` ([MoE-Eng] §6.3, §9
    ``routing = logits + self.route_bias``), or the logits alone.

    Reading: the softmax gate ranks the fp32 logits rather than the softmax
    probabilities of [MoE-Eng] §4.1; softmax is monotone, so the selected set is
    the same, and the choice keeps the decision free of any exp implementation.
    """
    keys = logits.astype(F32)
    if bias is not None:
        keys = (keys + bias.astype(F32)[None, :]).astype(F32)
    return keys


def topk_select(keys: np.ndarray, k: int) -> np.ndarray:
    """Per row, the ``k`` experts with the largest key, sorted by rank.

    Total order (reading; ``torch.topk`` leaves ties unspecified): larger key
    first, equal keys by lower expert index; -0.0 equals +0.0; NaN ranks below
    every number.  Returns int32 [N, k].
    """
    n, e = keys.shape
    if k > e:
        raise ValueError("top_k > n_experts")
    out = np.empty((n, k), dtype=np.int32)
    idx = np.arange(e)
    for t in range(n):
        row = keys[t].astype(np.float64)
        row = np.where(row == 0.0, 0.0, row)            # -0.0 -> +0.0
        nan = np.isnan(row)
        neg = np.where(nan, 0.0, -row)
        order = np.lexsort((idx, neg, nan))              # primary: not-NaN first
        out[t] = order[:k]
    return out


def _key_cmp(a, b):
    """Comparator of (key, expert) pairs for the brute-force top-K."""
    (ka, ia), (kb, ib) = a, b
    na, nb = np.isnan(ka), np.isnan(kb)
    if na != nb:
        return 1 if na else -1
    if not na and ka != kb:
        return -1 if ka > kb else 1
    return -1 if ia < ib else (1 if ia > ib else 0)


def topk_select_bruteforce(keys: np.ndarray, k: int) -> np.ndarray:
    """Brute force: sort every expert of a token with an explicit comparator."""
    n, e = keys.shape
    out = np.empty((n, k), dtype=np.int32)
    for t in range(n):
        pairs = [(float(keys[t, j]), j) for j in range(e)]
        pairs.sort(key=functools.cmp_to_key(_key_cmp))
        out[t] = [j for _, j in pairs[:k]]
    return out


def _sigmoid(v: np.ndarray, dtype=F32) -> np.ndarray:
    v = v.astype(dtype)
    return (dtype(1.0) / (dtype(1.0) + np.exp(-v))).astype(dtype)


def gate_weights(logits: np.ndarray, idx: np.ndarray, gate: str, dtype=F32) -> np.ndarray:
    """Renormalised gate weights of the selected experts, fp32 [N, K].

    softmax ([MoE-Eng] §4.1): ``p = softmax(logits)`` over all E, then
    ``p_sel / sum(p_sel)``.  sigmoid ([MoE-Eng] §4.3, §9): ``sigmoid`` of the
    *unbiased* selected logits, then ``s_sel / sum(s_sel)``.
    """
    lg = logits.astype(dtype)
    if gate == "softmax":
        m = lg.max(axis=1, keepdims=True)
        ex = np.exp((lg - m).astype(dtype)).astype(dtype)
        p = (ex / ex.sum(axis=1, keepdims=True, dtype=dtype)).astype(dtype)
        sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    elif gate == "sigmoid":
        sel = _sigmoid(np.take_along_axis(lg, idx.astype(np.int64), axis=1), dtype)
    else:
        raise ValueError(gate)
    return (sel / sel.sum(axis=1, keepdims=True, dtype=dtype)).astype(dtype)


def route(logits: np.ndarray, bias: np.ndarray | None, k: int, gate: str):
    """Top-K selection and renormalised weights from fp32 logits ([MoE-Eng] §9 step 1)."""
    idx = topk_select(selection_keys(logits, bias), k)
    return idx, gate_weights(logits, idx, gate)


# ----------------------------------------------------------------------------
# Histogram, offsets, permutation ([MoE-Eng] §9 load statistics, §12.5)
# ----------------------------------------------------------------------------
def histogram(idx: np.ndarray, n_exp: int) -> np.ndarray:
    """``counts[e]`` = number of token copies routed to expert e
    ([MoE-Eng] §9 ``load.scatter_add_``; §12.5 ``bincount``).  int32 [E]."""
    return np.bincount(idx.reshape(-1).astype(np.int64), minlength=n_exp).astype(np.int32)


def exclusive_offsets(counts: np.ndarray) -> np.ndarray:
    """``offsets[0] = 0``, ``offsets[e+1] = offsets[e] + counts[e]``.  int32 [E+1]."""
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    off[1:] = np.cumsum(counts.astype(np.int64))
    return off.astype(np.int32)


def permutation(idx: np.ndarray, n_exp: int):
    """Expert-major order of the token copies ([MoE-Eng] §12.5 sort by destination).

    Copy ``c = t*K + k``.  Rows are ordered by expert, then by ascending token
    (reading: the §9 loop's ``nonzero`` yields ascending tokens; a token reaches
    an expert at most once, so the order is total).  Returns ``row_of_copy``
    [N*K] and ``copy_of_row`` [N*K], both int32, inverse of each other.
    """
    flat = idx.reshape(-1)
    r = flat.shape[0]
    # Counting sort written out: walk the copies in token order and hand each
    # the next free row of its expert.
    counts = histogram(idx, n_exp)
    nxt = exclusive_offsets(counts)[:-1].astype(np.int64).copy()
    row_of_copy = np.empty(r, dtype=np.int32)
    for c in range(r):
        e = int(flat[c])
        row_of_copy[c] = nxt[e]
        nxt[e] += 1
    copy_of_row = np.empty(r, dtype=np.int32)
    copy_of_row[row_of_copy] = np.arange(r, dtype=np.int32)
    return row_of_copy, copy_of_row


# ----------------------------------------------------------------------------
# Experts ([MoE-Eng] §9 ``Expert``: w2(silu(w1 x) * w3 x), nn.Linear, no bias)
# ----------------------------------------------------------------------------
def _silu(a):
    return a / (1.0 + np.exp(-a))


def swiglu_expert(x, w1, w3, w2, dtype=F32):
    """One SwiGLU expert.  x [m, D]; w1, w3 [F, D]; w2 [D, F].

    Returns (y, a1, a3, h) with a1 = x w1^T, a3 = x w3^T, h = silu(a1) * a3,
    y = h w2^T, all in ``dtype``.
    """
    xx = x.astype(dtype)
    a1 = np.matmul(xx, w1.astype(dtype).T)
    a3 = np.matmul(xx, w3.astype(dtype).T)
    h = (_silu(a1) * a3).astype(dtype)
    y = np.matmul(h, w2.astype(dtype).T)
    return y, a1, a3, h


def moe_forward(x, logits, idx, g, w1, w3, w2, shared=None, dtype=F32):
    """Layer output by the loop over experts of [MoE-Eng] §9.

    For every expert: the tokens that chose it (``nonzero`` of the top-K mask,
    ascending token), their gate weight, the SwiGLU expert on the gathered rows,
    the weighted result added back at the token (``index_add_``).  Experts that
    no token chose are skipped.  The shared expert ([MoE-Eng] §5 formula;
    ``shared = (ws1, ws3, ws2)`` or None) is added to every token, ungated.

    ``logits`` is unused here; it is accepted so the call mirrors the layer.
    Returns ``(out [N, D], saved)``; ``saved`` keeps per-expert intermediates
    for :func:`moe_backward`.
    """
    del logits
    n, d = x.shape
    n_exp = w1.shape[0]
    out = np.zeros((n, d), dtype=dtype)
    saved = {"experts": {}, "shared": None}
    for e in range(n_exp):
        tok, kk = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        w = g[tok, kk].astype(dtype)[:, None]
        y, a1, a3, h = swiglu_expert(x[tok], w1[e], w3[e], w2[e], dtype)
        np.add.at(out, tok, y * w)
        saved["experts"][e] = (tok, kk, y, a1, a3, h)
    if shared is not None:
        ys, a1s, a3s, hs = swiglu_expert(x, shared[0], shared[1], shared[2], dtype)
        out = out + ys
        saved["shared"] = (ys, a1s, a3s, hs)
    return out, saved


# ----------------------------------------------------------------------------
# Capacity factor and token drop ([MoE-Eng] §6.4; §2.2 GShard): the
# comparison case of the dropless layer
# ----------------------------------------------------------------------------
def capacity(n_tok: int, n_exp: int, top_k: int, capacity_factor: float) -> int:
    """``capacity_factor * (tokens_per_batch / n_experts * top_k)`` ([MoE-Eng]
    §6.4), rounded up to whole token copies (reading)."""
    return int(np.ceil(capacity_factor * (n_tok / n_exp * top_k) - 1e-9))


def permutation_capacity(idx: np.ndarray, n_exp: int, cap: int):
    """Expert-major permutation with at most ``cap`` copies per expert: each
    expert keeps its first ``cap`` copies in token order (the order of the
    dropless permutation) and drops the rest (reading: overflow is dropped,
    [MoE-Eng] §6.4 "drop ... through the residual").

    Returns (row_of_copy with -1 for dropped copies, copy_of_row of the kept
    rows, kept counts, kept offsets [E+1], number of dropped copies)."""
    n, k = idx.shape
    roc_full, _ = permutation(idx, n_exp)
    off_full = exclusive_offsets(histogram(idx, n_exp))
    flat = idx.reshape(-1).astype(np.int64)
    rank = roc_full - off_full[flat]
    kept = np.minimum(histogram(idx, n_exp), cap).astype(np.int64)
    off = exclusive_offsets(kept)
    roc = np.where(rank < cap, off[flat] + rank, -1).astype(np.int64)
    cor = np.empty(int(kept.sum()), dtype=np.int64)
    keep = roc >= 0
    cor[roc[keep]] = np.nonzero(keep)[0]
    return roc, cor, kept, off, int((~keep).sum())


def moe_forward_capacity(x, logits, idx, g, w1, w3, w2, cap, shared=None, dtype=F32):
    """The layer forward with a per-expert capacity: as :func:`moe_forward`,
    but expert e processes only its first ``cap`` tokens (ascending token
    order) and a dropped copy contributes nothing to the combine (the token
    keeps only its residual path, outside the layer).  The gate weights of the
    kept copies are not renormalised.  Returns (out, saved) in the layout of
    :func:`moe_forward`, so :func:`moe_backward` gives the gradients: dropped
    copies get dg = 0 and still receive a router-logit gradient through the
    renormalisation of the kept ones."""
    n, d = x.shape
    xx = x.astype(dtype)
    out = np.zeros((n, d), dtype=dtype)
    saved = {"experts": {}}
    for e in range(w1.shape[0]):
        tok, kk = np.nonzero(idx == e)
        tok, kk = tok[:cap], kk[:cap]
        if tok.size == 0:
            continue
        y, a1, a3, h = swiglu_expert(xx[tok], w1[e], w3[e], w2[e], dtype)
        saved["experts"][e] = (tok, kk, y, a1, a3, h)
        np.add.at(out, tok, y * g[tok, kk].astype(dtype)[:, None])
    if shared is not None:
        ys, a1s, a3s, hs = swiglu_expert(xx, shared[0], shared[1], shared[2], dtype)
        saved["shared"] = (ys, a1s, a3s, hs)
        out = out + ys
    return out, saved


def moe_forward_dense_bruteforce(x, idx, g, w1, w3, w2, shared=None):
    """Pin for :func:`moe_forward`: evaluate every expert on every token in
    fp64, then sum the selected ones per token ([MoE-Eng] §5 formula
    ``y = shared(x) + sum_{i in TopK} gate_i * expert_i(x)``)."""
    n, d = x.shape
    n_exp = w1.shape[0]
    xx = x.astype(np.float64)
    all_y = np.empty((n_exp, n, d))
    for e in range(n_exp):
        all_y[e] = swiglu_expert(xx, w1[e], w3[e], w2[e], np.float64)[0]
    out = np.zeros((n, d))
    for t in range(n):
        for k in range(idx.shape[1]):
            out[t] += float(g[t, k]) * all_y[idx[t, k], t]
    if shared is not None:
        out += swiglu_expert(xx, shared[0], shared[1], shared[2], np.float64)[0]
    return out


# ----------------------------------------------------------------------------
# Backward (derivative of [MoE-Eng] §9 forward; §11.3 sparse backward)
# ----------------------------------------------------------------------------
def router_logit_grad(dg, g, logits, idx, gate, dtype=F32):
    """d(loss)/d(logits) [N, E] given d(loss)/d(g) for the selected weights.

    softmax + renorm: ``g_k = exp(l_k) / sum_sel exp(l_j)`` (the full-softmax
    denominator cancels), so ``dl_k = g_k (dg_k - sum_j g_j dg_j)`` on selected
    experts and 0 elsewhere.  sigmoid + renorm: ``g_k = s_k / S``, so
    ``dl_k = s_k (1 - s_k) / S * (dg_k - sum_j g_j dg_j)``.  The route bias only
    changes which experts are selected and receives no gradient ([MoE-Eng] §6.3).
    """
    n, n_exp = logits.shape
    dg = dg.astype(dtype)
    gg = g.astype(dtype)
    inner = (gg * dg).sum(axis=1, keepdims=True)
    if gate == "softmax":
        dsel = gg * (dg - inner)
    else:
        lsel = np.take_along_axis(logits, idx.astype(np.int64), axis=1).astype(dtype)
        s = 1.0 / (1.0 + np.exp(-lsel))
        ssum = s.sum(axis=1, keepdims=True)
        dsel = s * (1.0 - s) / ssum * (dg - inner)
    dl = np.zeros((n, n_exp), dtype=dtype)
    np.put_along_axis(dl, idx.astype(np.int64), dsel, axis=1)
    return dl


def moe_backward(dy, x, logits, idx, g, w_gate, w1, w3, w2, saved, gate,
                 shared=None, dtype=F32, train_router=True):
    """Gradients of the layer for an upstream gradient ``dy`` [N, D].

    Per expert e with rows ``tok`` (the forward's gathered tokens):
    ``dYw = g * dy[tok]``; ``dg = <dy[tok], y_e>``; ``dh = dYw w2_e``;
    ``da3 = dh * silu(a1)``; ``da1 = dh * a3 * s (1 + a1 (1 - s))`` with
    ``s = sigmoid(a1)``; ``dW2_e = dYw^T h``; ``dW1_e = da1^T x``;
    ``dW3_e = da3^T x``; ``dx[tok] += da1 w1_e + da3 w3_e``.  Experts with no
    token keep dW = 0 ([MoE-Eng] §11.3).  The shared expert is the same with
    gate 1 over all tokens.  Router: ``dlogits`` from :func:`router_logit_grad`,
    ``dW_g = dlogits^T x`` and ``dx += dlogits W_g``.

    Returns a dict with dx, dw1, dw3, dw2, dw_gate, dg, dlogits (and dws1,
    dws3, dws2 when a shared expert is present).
    """
    n, d = x.shape
    n_exp, f, _ = w1.shape
    k = idx.shape[1]
    xx = x.astype(dtype)
    dyy = dy.astype(dtype)
    dx = np.zeros((n, d), dtype=dtype)
    dw1 = np.zeros((n_exp, f, d), dtype=dtype)
    dw3 = np.zeros((n_exp, f, d), dtype=dtype)
    dw2 = np.zeros((n_exp, d, f), dtype=dtype)
    dg = np.zeros((n, k), dtype=dtype)

    def expert_bwd(dyw, xe, a1, a3, h, we1, we3, we2):
        dh = np.matmul(dyw, we2.astype(dtype))
        s = 1.0 / (1.0 + np.exp(-a1))
        da3 = dh * (a1 * s)
        da1 = dh * a3 * s * (1.0 + a1 * (1.0 - s))
        gw2 = np.matmul(dyw.T, h)
        gw1 = np.matmul(da1.T, xe)
        gw3 = np.matmul(da3.T, xe)
        gx = np.matmul(da1, we1.astype(dtype)) + np.matmul(da3, we3.astype(dtype))
        return gw1, gw3, gw2, gx

    for e, (tok, kk, y, a1, a3, h) in saved["experts"].items():
        dg[tok, kk] = (dyy[tok] * y).sum(axis=1)
        dyw = dyy[tok] * g[tok, kk].astype(dtype)[:, None]
        gw1, gw3, gw2, gx = expert_bwd(dyw, xx[tok], a1, a3, h, w1[e], w3[e], w2[e])
        dw1[e], dw3[e], dw2[e] = gw1, gw3, gw2
        np.add.at(dx, tok, gx)

    res = {}
    if shared is not None:
        ys, a1s, a3s, hs = saved["shared"]
        gw1, gw3, gw2, gx = expert_bwd(dyy, xx, a1s, a3s, hs, shared[0], shared[1], shared[2])
        res.update(dws1=gw1, dws3=gw3, dws2=gw2)
        dx = dx + gx

    dl = router_logit_grad(dg, g, logits, idx, gate, dtype)
    dw_gate = np.matmul(dl.T, xx)
    if train_router:
        dx = dx + np.matmul(dl, w_gate.astype(dtype))
    res.update(dx=dx, dw1=dw1, dw3=dw3, dw2=dw2, dw_gate=dw_gate, dg=dg, dlogits=dl)
    return res


# ----------------------------------------------------------------------------
# Load statistics and balancing ([MoE-Eng] §6.2, §6.3, §9, §13.9)
# ----------------------------------------------------------------------------
def load_stat(counts: np.ndarray) -> np.ndarray:
    """``load / load.sum()`` in fp32 ([MoE-Eng] §9 step 4)."""
    load = counts.astype(F32)
    return (load / load.sum(dtype=F32)).astype(F32)


def update_bias(counts: np.ndarray, bias: np.ndarray, gamma: float = 1e-3,
                mode: int = 0, target: float | None = None) -> np.ndarray:
    """Online route-bias update ([MoE-Eng] §9 ``update_balance_bias``; §6.3 prose).

    mode 0 (the listing): ``bias -= gamma * sign(load_stat - target) *
    max(load_stat, 1e-6)``, all fp32, ``target = 1/E`` by default, the window
    being the last batch.  mode 1 (the prose of §6.3): ``bias -= gamma *
    sign(load_stat - target)``, i.e. minus gamma when over-loaded, plus gamma
    when under-loaded.  Reading: an empty batch (no copies) leaves the bias
    unchanged (the listing would divide 0 by 0).  Returns the new bias (fp32).
    """
    bias = bias.astype(F32).copy()
    if int(counts.astype(np.int64).sum()) == 0:
        return bias
    ls = load_stat(counts)
    tgt = F32(1.0 / len(counts)) if target is None else F32(target)
    sgn = np.sign((ls - tgt).astype(F32)).astype(F32)
    step = (F32(gamma) * sgn).astype(F32)
    if mode == 0:
        step = (step * np.maximum(ls, F32(1e-6))).astype(F32)
    elif mode != 1:
        raise ValueError(mode)
    return (bias - step).astype(F32)


def aux_loss(logits: np.ndarray, idx: np.ndarray, n_exp: int, gate: str = "softmax") -> float:
    """GShard-style auxiliary loss of [MoE-Eng] §6.2: ``E * sum_i f_i P_i``.

    ``f_i`` = mean over tokens of the top-K mask (so ``sum f = K``), ``P_i`` =
    mean gate probability.  For the softmax gate P is the softmax over all
    experts; for the sigmoid gate (reading: the pages give no P for it) the
    per-token sigmoid scores normalised over all experts.  Value only (fp64).
    """
    lg = logits.astype(np.float64)
    if gate == "softmax":
        ex = np.exp(lg - lg.max(axis=1, keepdims=True))
        probs = ex / ex.sum(axis=1, keepdims=True)
    else:
        s = 1.0 / (1.0 + np.exp(-lg))
        probs = s / s.sum(axis=1, keepdims=True)
    mask = np.zeros_like(probs)
    np.put_along_axis(mask, idx.astype(np.int64), 1.0, axis=1)
    f = mask.mean(axis=0)
    p = probs.mean(axis=0)
    return float(n_exp * (f * p).sum())


def aux_loss_grad(logits: np.ndarray, idx: np.ndarray, n_exp: int, gate: str = "softmax") -> np.ndarray:
    """Gradient of :func:`aux_loss` with respect to the logits [N, E] (fp64),
    the top-K fractions ``f`` held fixed (they come from the discrete
    selection).  With ``P_i = mean_t q_{t,i}``:

    * softmax: ``q = softmax(l)``, ``dq_i/dl_j = q_i (delta_ij - q_j)``, so
      ``d aux / d l_{t,j} = E/N * q_{t,j} (f_j - sum_i f_i q_{t,i})``;
    * sigmoid: ``q_i = s_i / S`` with ``s = sigmoid(l)``, ``S = sum s``, so
      ``d aux / d l_{t,j} = E/N * s_j (1 - s_j) / S * (f_j - sum_i f_i q_{t,i})``.
    """
    lg = logits.astype(np.float64)
    n = lg.shape[0]
    mask = np.zeros_like(lg)
    np.put_along_axis(mask, idx.astype(np.int64), 1.0, axis=1)
    f = mask.mean(axis=0)
    if gate == "softmax":
        ex = np.exp(lg - lg.max(axis=1, keepdims=True))
        q = ex / ex.sum(axis=1, keepdims=True)
        dq = q
    else:
        sg = 1.0 / (1.0 + np.exp(-lg))
        ssum = sg.sum(axis=1, keepdims=True)
        q = sg / ssum
        dq = sg * (1.0 - sg) / ssum
    inner = (q * f[None, :]).sum(axis=1, keepdims=True)
    return n_exp / n * dq * (f[None, :] - inner)


def monitor_stats(history: list[np.ndarray], last: int = 100) -> dict:
    """Monitor hook of [MoE-Eng] §13.9 over a list of ``load_stat`` vectors:
    mean of the last ``last`` entries, then its minimum, its entropy
    ``-sum r log(r + 1e-9)`` and the number of experts under ``0.3 / E``."""
    recent = np.stack(history[-last:]).astype(np.float64).mean(axis=0)
    entropy = float(-(recent * np.log(recent + 1e-9)).sum())
    cold = int((recent < 0.3 / len(recent)).sum())
    return {"min_load": float(recent.min()), "entropy": entropy, "cold_experts": cold}
