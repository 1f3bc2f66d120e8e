"""Pins of the CPU oracle against things other than itself: worked examples,
closed forms, invariants, brute force on tiny inputs, special cases that
reduce to plain dense computations, fp64 finite differences and an
independent autograd derivation.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(a):
    """Round an fp32 array to bf16 values (kept as fp32), round to nearest even."""
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _layer(n, d, f, e, k, gate="softmax", bias=False, shared=0, seed=0, wscale=0.3):
    r = _rng(seed)
    p = {
        "x": _bf16(r.standard_normal((n, d))),
        "w_gate": _bf16(r.standard_normal((e, d)) * wscale),
        "w1": _bf16(r.standard_normal((e, f, d)) * wscale),
        "w3": _bf16(r.standard_normal((e, f, d)) * wscale),
        "w2": _bf16(r.standard_normal((e, d, f)) * wscale),
        "bias": (r.standard_normal(e).astype(np.float32) * 0.5) if bias else None,
        "shared": None,
    }
    if shared:
        p["shared"] = (_bf16(r.standard_normal((shared, d)) * wscale),
                       _bf16(r.standard_normal((shared, d)) * wscale),
                       _bf16(r.standard_normal((d, shared)) * wscale))
    return p


# ---------------------------------------------------------------- router ---
def test_router_worked_examples():
    ex = json.load(open(os.path.join(GOLD, "router_worked_examples.json")))
    for c in ex["cases"]:
        lg = np.array(c["logits"], dtype=np.float32)
        bias = None if c["bias"] is None else np.array(c["bias"], dtype=np.float32)
        idx, g = O.route(lg, bias, c["k"], c["gate"])
        assert idx.tolist() == c["idx"], c["name"]
        np.testing.assert_allclose(g, np.array(c["g"]), rtol=2e-7, atol=0, err_msg=c["name"])


@pytest.mark.parametrize("e,k", [(8, 2), (16, 4), (64, 8), (5, 5)])
def test_topk_matches_bruteforce(e, k):
    r = _rng(e * 10 + k)
    keys = r.standard_normal((200, e)).astype(np.float32)
    keys[:50] = np.round(keys[:50])                     # many exact ties
    keys[50:60, 0] = -0.0
    keys[50:60, 1] = 0.0
    keys[60:65, 2] = np.nan
    keys[65:70] = np.nan                                  # a whole row of NaN
    np.testing.assert_array_equal(O.topk_select(keys, k), O.topk_select_bruteforce(keys, k))


def test_topk_zero_gate_picks_first_k_with_equal_weights():
    # W_g = 0 -> every logit is 0 -> experts 0..K-1, each weight exactly 1/K
    x = np.ones((7, 16), dtype=np.float32)
    lg = O.gate_logits(x, np.zeros((8, 16), dtype=np.float32))
    for gate in ("softmax", "sigmoid"):
        idx, g = O.route(lg, None, 4, gate)
        assert (idx == np.arange(4)).all()
        assert (g == np.float32(0.25)).all()


def test_gate_weights_sum_to_one():
    r = _rng(3)
    lg = (r.standard_normal((500, 32)) * 3).astype(np.float32)
    for gate in ("softmax", "sigmoid"):
        idx, g = O.route(lg, None, 6, gate)
        s = g.astype(np.float64).sum(axis=1)
        assert np.abs(s - 1.0).max() <= 4 * np.finfo(np.float32).eps


def test_softmax_renorm_equals_softmax_over_selected():
    # full-softmax then renorm == softmax restricted to the selected logits
    r = _rng(4)
    lg = (r.standard_normal((300, 16)) * 2).astype(np.float32)
    idx, g = O.route(lg, None, 3, "softmax")
    sel = np.take_along_axis(lg.astype(np.float64), idx.astype(np.int64), axis=1)
    ref = np.exp(sel - sel.max(axis=1, keepdims=True))
    ref /= ref.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(g, ref, rtol=1e-6, atol=1e-7)


def test_bias_changes_selection_not_weights():
    r = _rng(5)
    lg = r.standard_normal((100, 8)).astype(np.float32)
    bias = np.array([5, 0, 0, 0, 0, 0, 0, -5], dtype=np.float32)
    idx, g = O.route(lg, bias, 2, "sigmoid")
    assert (idx[:, 0] == 0).all() and not (idx == 7).any()
    s = 1 / (1 + np.exp(-np.take_along_axis(lg.astype(np.float64), idx.astype(np.int64), axis=1)))
    np.testing.assert_allclose(g, s / s.sum(axis=1, keepdims=True), rtol=1e-6)


# ------------------------------------------------ histogram / permutation ---
@pytest.mark.parametrize("n,e,k", [(256, 8, 2), (300, 64, 8), (1, 4, 4), (50, 16, 1)])
def test_histogram_offsets_permutation_invariants(n, e, k):
    r = _rng(n + e)
    lg = r.standard_normal((n, e)).astype(np.float32)
    lg[:, 0] += 1.0                                        # skew
    idx, _ = O.route(lg, None, k, "softmax")
    counts = O.histogram(idx, e)
    off = O.exclusive_offsets(counts)
    assert counts.sum() == n * k and off[0] == 0 and off[-1] == n * k
    roc, cor = O.permutation(idx, e)
    assert sorted(roc.tolist()) == list(range(n * k))      # bijection
    assert (cor[roc] == np.arange(n * k)).all()            # inverse maps
    flat = idx.reshape(-1)
    for ex in range(e):
        rows = np.arange(off[ex], off[ex + 1])
        assert (flat[cor[rows]] == ex).all()               # expert-major
        toks = cor[rows] // k
        assert (np.diff(toks) > 0).all()                   # ascending token
    # same order as a library stable sort by expert of the copies
    assert (cor == np.argsort(flat, kind="stable")).all()


# --------------------------------------------------------------- forward ---
@pytest.mark.parametrize("gate,bias,shared", [("softmax", False, 0), ("sigmoid", True, 24)])
def test_forward_matches_dense_bruteforce(gate, bias, shared):
    p = _layer(40, 16, 24, 6, 2, gate, bias, shared, seed=7)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, p["bias"], 2, gate)
    out, _ = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], p["shared"], dtype=np.float64)
    ref = O.moe_forward_dense_bruteforce(p["x"], idx, g, p["w1"], p["w3"], p["w2"], p["shared"])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    out32, _ = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], p["shared"])
    assert np.linalg.norm(out32 - ref) / np.linalg.norm(ref) < 1e-5


def test_forward_single_expert_is_dense_swiglu():
    # E = 1, K = 1: the layer is a plain SwiGLU FFN (torch fp64 matmuls)
    p = _layer(33, 16, 40, 1, 1, seed=8)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, None, 1, "softmax")
    assert (g == 1).all()
    out, _ = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], dtype=np.float64)
    x = torch.from_numpy(p["x"]).double()
    a1 = x @ torch.from_numpy(p["w1"][0]).double().T
    a3 = x @ torch.from_numpy(p["w3"][0]).double().T
    ref = (torch.nn.functional.silu(a1) * a3) @ torch.from_numpy(p["w2"][0]).double().T
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_forward_all_tokens_one_expert():
    p = _layer(20, 8, 16, 5, 1, gate="sigmoid", seed=9)
    bias = np.array([0, 0, 0, 1e4, 0], dtype=np.float32)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, bias, 1, "sigmoid")
    assert (idx == 3).all() and (g == 1).all()
    counts = O.histogram(idx, 5)
    assert counts.tolist() == [0, 0, 0, 20, 0]
    out, _ = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], dtype=np.float64)
    ref = O.swiglu_expert(p["x"], p["w1"][3], p["w3"][3], p["w2"][3], np.float64)[0]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_forward_k_equals_e_is_soft_moe():
    # softmax with K = E: every expert weighted by its full-softmax probability
    p = _layer(16, 8, 12, 4, 4, seed=10)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, None, 4, "softmax")
    out, _ = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], dtype=np.float64)
    probs = torch.softmax(torch.from_numpy(lg).double(), dim=1).numpy()
    ref = np.zeros_like(out)
    for e in range(4):
        ref += probs[:, e:e + 1] * O.swiglu_expert(p["x"], p["w1"][e], p["w3"][e], p["w2"][e], np.float64)[0]
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)


# -------------------------------------------------------------- backward ---
def _loss_and_grads(p, dy, gate, k, idx_frozen=None, dtype=np.float64):
    lg = O.gate_logits(p["x"], p["w_gate"], dtype)
    if idx_frozen is None:
        idx = O.topk_select(O.selection_keys(lg.astype(np.float32), p["bias"]), k)
    else:
        idx = idx_frozen
    g = O.gate_weights(lg, idx, gate, dtype)
    out, saved = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], p["shared"], dtype=dtype)
    loss = float((out * dy).sum())
    return loss, idx, lg, g, saved


@pytest.mark.parametrize("gate,shared", [("softmax", 0), ("sigmoid", 6)])
def test_backward_finite_differences(gate, shared):
    n, d, f, e, k = 16, 8, 16, 4, 2
    p = _layer(n, d, f, e, k, gate, bias=(gate == "sigmoid"), shared=shared, seed=11, wscale=0.5)
    for key in ("x", "w_gate", "w1", "w3", "w2"):
        p[key] = p[key].astype(np.float64)
    if shared:
        p["shared"] = tuple(a.astype(np.float64) for a in p["shared"])
    dy = _rng(12).standard_normal((n, d))
    loss, idx, lg, g, saved = _loss_and_grads(p, dy, gate, k)
    keys = np.sort(O.selection_keys(lg.astype(np.float32), p["bias"]), axis=1)
    assert (keys[:, -k] - keys[:, -k - 1]).min() > 1e-3      # routing margin >> h
    gr = O.moe_backward(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved,
                        gate, p["shared"], dtype=np.float64)
    h = 1e-6
    r = _rng(13)
    targets = [("x", "dx"), ("w_gate", "dw_gate"), ("w1", "dw1"), ("w3", "dw3"), ("w2", "dw2")]
    if shared:
        targets += [(("shared", 0), "dws1"), (("shared", 1), "dws3"), (("shared", 2), "dws2")]
    for src, gname in targets:
        arr = p[src] if isinstance(src, str) else p["shared"][src[1]]
        for _ in range(6):
            pos = tuple(int(r.integers(s)) for s in arr.shape)
            old = arr[pos]
            arr[pos] = old + h
            lp = _loss_and_grads(p, dy, gate, k, idx)[0]
            arr[pos] = old - h
            lm = _loss_and_grads(p, dy, gate, k, idx)[0]
            arr[pos] = old
            fd = (lp - lm) / (2 * h)
            an = gr[gname][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (gname, pos, fd, an)


def _torch_layer_restatement(x, w_gate, w1, w3, w2, bias, k, gate, shared):
    """The page's single-GPU MoE layer forward written with torch ops
    (fp64 CPU), used only to get gradients from autograd."""
    logits = x @ w_gate.T
    routing = logits + (bias if bias is not None else 0)
    _, topk_idx = routing.topk(k, dim=-1)
    if gate == "sigmoid":
        gw = torch.sigmoid(logits.gather(-1, topk_idx))
    else:
        gw = torch.softmax(logits, dim=-1).gather(-1, topk_idx)
    gw = gw / gw.sum(-1, keepdim=True)
    out = torch.zeros_like(x)
    for e in range(w1.shape[0]):
        mask = topk_idx == e
        if not mask.any():
            continue
        tok, kk = mask.nonzero(as_tuple=True)
        xs = x[tok]
        y = (torch.nn.functional.silu(xs @ w1[e].T) * (xs @ w3[e].T)) @ w2[e].T
        out = out.index_add(0, tok, y * gw[tok, kk].unsqueeze(-1))
    if shared is not None:
        out = out + (torch.nn.functional.silu(x @ shared[0].T) * (x @ shared[1].T)) @ shared[2].T
    return out, topk_idx


@pytest.mark.parametrize("gate,shared", [("softmax", 0), ("sigmoid", 10)])
def test_backward_matches_autograd(gate, shared):
    n, d, f, e, k = 24, 12, 20, 6, 3
    p = _layer(n, d, f, e, k, gate, bias=(gate == "sigmoid"), shared=shared, seed=14, wscale=0.4)
    dy = _rng(15).standard_normal((n, d))
    lg = O.gate_logits(p["x"], p["w_gate"], np.float64)
    idx = O.topk_select(O.selection_keys(lg.astype(np.float32), p["bias"]), k)
    g = O.gate_weights(lg, idx, gate, np.float64)
    out, saved = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], p["shared"], dtype=np.float64)
    gr = O.moe_backward(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved, gate,
                        p["shared"], dtype=np.float64)
    T = {key: torch.tensor(p[key], dtype=torch.float64, requires_grad=True)
         for key in ("x", "w_gate", "w1", "w3", "w2")}
    sh = None
    if shared:
        sh = tuple(torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in p["shared"])
    b = None if p["bias"] is None else torch.tensor(p["bias"], dtype=torch.float64)
    tout, tidx = _torch_layer_restatement(T["x"], T["w_gate"], T["w1"], T["w3"], T["w2"], b, k, gate, sh)
    assert np.array_equal(np.sort(tidx.numpy(), 1), np.sort(idx, 1))
    np.testing.assert_allclose(tout.detach().numpy(), out, rtol=1e-10, atol=1e-12)
    (tout * torch.from_numpy(dy)).sum().backward()
    for key, gname in [("x", "dx"), ("w_gate", "dw_gate"), ("w1", "dw1"), ("w3", "dw3"), ("w2", "dw2")]:
        np.testing.assert_allclose(gr[gname], T[key].grad.numpy(), rtol=1e-9, atol=1e-10, err_msg=gname)
    if shared:
        for i, gname in enumerate(("dws1", "dws3", "dws2")):
            np.testing.assert_allclose(gr[gname], sh[i].grad.numpy(), rtol=1e-9, atol=1e-10)


def test_backward_unused_expert_has_zero_grad():
    p = _layer(10, 8, 8, 4, 1, gate="sigmoid", seed=16)
    bias = np.array([1e4, 0, 0, 0], dtype=np.float32)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, bias, 1, "sigmoid")
    out, saved = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"])
    gr = O.moe_backward(np.ones_like(out), p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"],
                        saved, "sigmoid")
    for e in (1, 2, 3):
        assert not gr["dw1"][e].any() and not gr["dw3"][e].any() and not gr["dw2"][e].any()
    # K = 1 with renorm: g == 1 regardless of the logit, so the router gets no gradient
    assert not gr["dlogits"].any()


# ------------------------------------------------- balancing / monitoring ---
def test_bias_update_worked_example():
    ex = json.load(open(os.path.join(GOLD, "bias_update_worked_example.json")))
    counts = np.array(ex["counts"], dtype=np.int32)
    b0 = np.array(ex["bias_in"], dtype=np.float32)
    np.testing.assert_array_equal(O.load_stat(counts), np.array(ex["load_stat"], dtype=np.float32))
    np.testing.assert_allclose(O.update_bias(counts, b0, ex["gamma"], 0),
                               np.array(ex["mode0_bias_out"], dtype=np.float32), rtol=3e-7, atol=0)  # fp32 products: a few ulp
    np.testing.assert_allclose(O.update_bias(counts, b0, ex["gamma"], 1),
                               np.array(ex["mode1_bias_out"], dtype=np.float32), rtol=1e-7, atol=0)


def test_bias_update_balanced_and_empty():
    b = np.full(4, 0.5, dtype=np.float32)
    assert (O.update_bias(np.array([2, 2, 2, 2]), b) == b).all()   # exactly balanced: no step
    assert (O.update_bias(np.zeros(4, dtype=np.int32), b) == b).all()


def test_aux_loss_closed_forms():
    # W_g = 0: P = 1/E everywhere, the top-K mask picks experts 0..K-1: loss = K
    lg = np.zeros((64, 8), dtype=np.float32)
    idx = O.topk_select(lg, 2)
    assert O.aux_loss(lg, idx, 8) == pytest.approx(2.0, abs=1e-12)
    # K = 1 with perfectly uniform hard routing and uniform probabilities: loss = 1
    idx1 = (np.arange(64) % 8).reshape(64, 1)
    assert O.aux_loss(lg, idx1, 8) == pytest.approx(1.0, abs=1e-12)


def test_monitor_stats_hand_example():
    h = [np.array([0.5, 0.3, 0.2, 0.0]), np.array([0.3, 0.3, 0.3, 0.1])]
    st = O.monitor_stats(h)
    recent = np.array([0.4, 0.3, 0.25, 0.05])
    assert st["min_load"] == pytest.approx(0.05)
    assert st["cold_experts"] == 1                      # 0.05 < 0.3/4
    assert st["entropy"] == pytest.approx(-sum(r * math.log(r + 1e-9) for r in recent))


# ---------------------------------------------------------------- MXFP8 ---
def test_e4m3_table_and_rounding():
    t = json.load(open(os.path.join(GOLD, "e4m3_table.json")))
    for code, val in t["codes"].items():
        got = O.e4m3_decode(np.array([int(code, 16)]))[0]
        assert got == val and np.signbit(got) == np.signbit(val), code
    for code in t["nan_codes"]:
        assert np.isnan(O.e4m3_decode(np.array([int(code, 16)]))[0])
    for v, code in t["round_cases"]:
        assert int(O.e4m3_encode(np.array([v]))[0]) == int(code, 16), v


def test_e4m3_roundtrip_all_codes_and_nearest():
    codes = np.arange(256)
    vals = O.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert (O.e4m3_encode(vals[finite]) == codes[finite]).all()
    # brute force: every encoded value is a nearest representable value
    grid = np.unique(vals[finite])
    r = _rng(17)
    xs = np.concatenate([r.standard_normal(2000) * 50, r.standard_normal(2000) * 0.01])
    enc = O.e4m3_decode(O.e4m3_encode(xs))
    clipped = np.clip(xs, -448, 448)
    best = np.abs(grid[None, :] - clipped[:, None]).min(axis=1)
    assert np.allclose(np.abs(enc - clipped), best, rtol=0, atol=0)


def test_mx_scale_is_the_unique_power_of_two():
    r = _rng(18)
    amax = np.abs(r.standard_normal(500)) * 10.0 ** r.integers(-20, 20, 500)
    ex = O.e8m0_scale_exponent(amax)
    for a, e in zip(amax, ex):
        # brute force over exponents: the one with 2^8 <= amax / 2^e < 2^9
        cands = [j for j in range(-127, 128) if 256 <= a / 2.0 ** j < 512]
        assert cands == [e]


def test_mx_quantize_group_aware_blocks():
    r = _rng(19)
    x = r.standard_normal((70, 3))
    codes, scales, starts = O.mx_quantize(x, axis=0, group_starts=[0, 40, 45])
    assert starts == [0, 32, 40, 45]
    deq = O.mx_dequantize(codes, scales, starts, axis=0)
    assert np.abs(deq - x).max() <= np.abs(x).max() * 2 ** -3


def test_mx_fake_quant_properties():
    r = _rng(20)
    # rows spanning 2^-20 .. 2^20 in magnitude: blocks along the right axis keep
    # every row's error within its own scale: half an E4M3 step (2^-4) of each
    # element, except a block maximum in [448, 512) * 2^e, which saturates to
    # 448 * 2^e (at most 1/8 of the row maximum)
    x = r.standard_normal((16, 96)) * np.exp2(np.linspace(-20, 20, 16))[:, None]
    fq = O.mx_fake_quant(x, axis=1)
    rel_rows = np.abs(fq - x).max(axis=1) / np.abs(x).max(axis=1)
    assert (rel_rows <= 0.125).all()
    wrong = O.mx_fake_quant(x, axis=0)           # blocks across rows lose the small rows
    assert (np.abs(wrong - x).max(axis=1) / np.abs(x).max(axis=1)).max() > 0.5
    assert np.array_equal(O.mx_fake_quant(fq, axis=1), fq)              # idempotent
    assert np.array_equal(O.mx_fake_quant(x * 2.0 ** 7, axis=1), fq * 2.0 ** 7)   # power-of-two scale invariance


def test_mxfp8_forward_reduces_to_exact_on_representable_operands():
    """With x and weights already MXFP8-representable and h quantisation the
    only rounding left, the quantisation-aware layer differs from the fp64
    dense brute force by at most h's quantisation (relative 2^-4 per element)."""
    p = _layer(24, 64, 64, 4, 2, seed=21)
    for key in ("x", "w1", "w3", "w2"):
        axis = 1 if p[key].ndim == 2 else 2
        p[key] = O.mx_fake_quant(p[key], axis=axis).astype(np.float32)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, None, 2, "softmax")
    out = O.moe_forward_mxfp8(p["x"], idx, g, p["w1"], p["w3"], p["w2"])
    ref = O.moe_forward_dense_bruteforce(p["x"], idx, g, p["w1"], p["w3"], p["w2"])
    e = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert 1e-4 < e < 6e-2          # h quantisation is visible, and bounded


# ------------------------------------------------------- MXFP8 backward ---
def _mx_case(seed, gate="sigmoid", shared=64):
    p = _layer(40, 64, 96, 4, 2, gate=gate, bias=gate == "sigmoid", shared=shared, seed=seed)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, p["bias"], 2, gate)
    dy = _bf16(_rng(seed + 100).standard_normal(p["x"].shape))
    return p, lg, idx, g, dy


def test_mxfp8_backward_with_identity_quantiser_is_the_bf16_backward():
    """Wiring pin: with the quantiser replaced by the identity every GEMM of
    the MXFP8 backward is the plain fp32 product, so the result must be the
    (finite-difference-pinned) bf16 oracle's backward on the same saved
    activations."""
    p, lg, idx, g, dy = _mx_case(31)
    _, saved = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], p["shared"])
    ref = O.moe_backward(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved, "sigmoid",
                         p["shared"])
    ident = lambda a, axis=None: np.asarray(a, np.float64)   # noqa: E731
    got = O.moe_backward_mxfp8(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved, "sigmoid",
                               p["shared"], quant=ident, store=ident)
    for key in ("dx", "dw1", "dw3", "dw2", "dw_gate", "dg", "dlogits", "dws1", "dws3", "dws2"):
        assert np.allclose(got[key], ref[key], rtol=1e-5, atol=1e-5 * np.abs(ref[key]).max()), key


def _block_scaled_product(a, b, starts):
    """sum_r a[r, i] b[r, j] with both operands quantised along r: per block,
    the products of the decoded E4M3 codes times 2^(scale_a + scale_b)."""
    ca, sa, st = O.mx_quantize(a, axis=0, group_starts=starts)
    cb, sb, _ = O.mx_quantize(b, axis=0, group_starts=starts)
    va, vb = O.e4m3_decode(ca), O.e4m3_decode(cb)
    ends = list(st[1:]) + [a.shape[0]]
    out = np.zeros((a.shape[1], b.shape[1]))
    for blk, (lo, hi) in enumerate(zip(st, ends)):
        part = va[lo:hi].T @ vb[lo:hi]
        out += part * np.exp2(sa[blk].astype(np.float64) - 127)[:, None] * np.exp2(sb[blk].astype(np.float64) - 127)[None, :]
    return out


def test_mxfp8_backward_weight_gradients_are_group_aware_block_products():
    """Axis pin: dW2 of every expert equals the block-scaled product of dYw and
    h quantised along the tokens of the whole expert-major permuted buffer
    with blocks restarting at each expert's first row (``group_starts``), and
    dh-side gradients differ from the ones with blocks across experts."""
    p, lg, idx, g, dy = _mx_case(32, shared=0)
    out, saved = O.moe_forward_mxfp8(p["x"], idx, g, p["w1"], p["w3"], p["w2"], None, return_saved=True)
    res = O.moe_backward_mxfp8(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved, "sigmoid")
    exps = sorted(saved["experts"])
    # dYw as the layer stores it (bf16), h as saved
    dyw = np.concatenate([O.bf16_round(dy[saved["experts"][e][0]] * g[saved["experts"][e][0], saved["experts"][e][1]][:, None])
                          for e in exps])
    hh = np.concatenate([saved["experts"][e][5] for e in exps])
    sizes = [len(saved["experts"][e][0]) for e in exps]
    starts = list(np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(int))
    assert any(s % 32 for s in starts)      # some expert starts off a 32-row boundary
    lo = 0
    for e, m in zip(exps, sizes):
        want = _block_scaled_product(dyw[lo:lo + m], hh[lo:lo + m], [0])
        assert np.allclose(res["dw2"][e], want, rtol=1e-5, atol=1e-6 * np.abs(want).max()), e
        lo += m
    # blocks taken across the whole buffer (ignoring expert boundaries) give other values
    whole = _block_scaled_product(dyw, hh, list(range(0, len(dyw), 32)))
    per_expert = sum(res["dw2"][e] for e in exps)
    assert not np.allclose(whole, per_expert, rtol=1e-4)


def test_mxfp8_backward_error_is_bounded_and_visible():
    """Against the fp32 backward of the fp32 forward, the MXFP8 backward
    differs by the quantisation of its GEMM operands: visible (> 1e-3) and
    bounded (< 0.1 normwise) for every gradient."""
    p, lg, idx, g, dy = _mx_case(33)
    _, saved_q = O.moe_forward_mxfp8(p["x"], idx, g, p["w1"], p["w3"], p["w2"], p["shared"], return_saved=True)
    got = O.moe_backward_mxfp8(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved_q, "sigmoid",
                               p["shared"])
    _, saved = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], p["shared"])
    ref = O.moe_backward(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved, "sigmoid",
                         p["shared"])
    for key in ("dx", "dw1", "dw3", "dw2", "dws1", "dws2"):
        e = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert 1e-3 < e < 0.1, (key, e)


def test_bf16_round_is_round_to_nearest_even():
    """The oracle's bf16 storage rounding against torch's fp32 -> bf16
    conversion (round to nearest even), including exact ties."""
    r = _rng(34)
    v = np.concatenate([r.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** r.integers(-30, 30, 20000),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0], np.float32)])
    want = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    got = O.bf16_round(v)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_mx_quantize_block_vectorised_path_equals_block_loop():
    """The all-blocks-at-once path (no group boundaries, whole blocks) against
    the block-by-block path (forced through group_starts=[0])."""
    r = _rng(35)
    x = r.standard_normal((5, 7, 96)) * np.exp2(r.integers(-40, 40, (5, 7, 1)))
    for axis in (2, 0):
        xa = np.moveaxis(x, 2, axis) if axis == 0 else x
        c1, s1, st1 = O.mx_quantize(xa, axis=axis if axis == 2 else 0)
        c2, s2, st2 = O.mx_quantize(xa, axis=axis if axis == 2 else 0, group_starts=[0])
        assert st1 == st2 and np.array_equal(c1, c2) and np.array_equal(s1, s2)
        assert np.array_equal(O.mx_dequantize(c1, s1, st1, axis=axis if axis == 2 else 0),
                              O.mx_dequantize(c2, s2, [0] + st2[1:], axis=axis if axis == 2 else 0))


@pytest.mark.parametrize("gate", ["softmax", "sigmoid"])
def test_aux_loss_grad_matches_finite_differences(gate):
    """The aux-loss logit gradient against fp64 central differences of the
    aux-loss value with the top-K selection held fixed."""
    r = _rng(36)
    n, e, k = 12, 6, 2
    lg = r.standard_normal((n, e))
    idx = O.topk_select(O.selection_keys(lg.astype(np.float32), None), k)
    grad = O.aux_loss_grad(lg, idx, e, gate)
    h = 1e-6
    fd = np.zeros_like(lg)
    for t in range(n):
        for j in range(e):
            lp, lm = lg.copy(), lg.copy()
            lp[t, j] += h
            lm[t, j] -= h
            fd[t, j] = (O.aux_loss(lp, idx, e, gate) - O.aux_loss(lm, idx, e, gate)) / (2 * h)
    assert np.allclose(grad, fd, rtol=1e-6, atol=1e-9)
    assert abs(grad.sum()) < 1e-9 if gate == "softmax" else True   # softmax: invariant to a per-token shift


# ------------------------------------------------- capacity factor / drop ---
def test_capacity_formula():
    """capacity = cf * (tokens / experts * top_k), rounded up to whole copies."""
    assert O.capacity(4096, 8, 2, 1.0) == 1024
    assert O.capacity(4096, 256, 8, 1.25) == 160
    assert O.capacity(100, 8, 2, 1.0) == 25
    assert O.capacity(10, 3, 1, 1.0) == 4          # 3.33 -> 4


def test_capacity_hand_example():
    """Ten tokens, K = 1, E = 2: tokens 0-7 pick expert 0, tokens 8-9 expert 1.
    cf = 1 -> capacity 5: expert 0 keeps tokens 0-4, drops 5-7."""
    idx = np.array([[0]] * 8 + [[1]] * 2, dtype=np.int32)
    cap = O.capacity(10, 2, 1, 1.0)
    roc, cor, kept, off, dropped = O.permutation_capacity(idx, 2, cap)
    assert cap == 5 and dropped == 3
    assert roc.tolist() == [0, 1, 2, 3, 4, -1, -1, -1, 5, 6]
    assert cor.tolist() == [0, 1, 2, 3, 4, 8, 9]
    assert kept.tolist() == [5, 2] and off.tolist() == [0, 5, 7]


def test_capacity_large_factor_is_dropless():
    p = _layer(40, 16, 24, 4, 2, seed=41)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, None, 2, "softmax")
    cap = int(O.histogram(idx, 4).max())
    roc, cor, kept, off, dropped = O.permutation_capacity(idx, 4, cap)
    roc0, cor0 = O.permutation(idx, 4)
    assert dropped == 0 and np.array_equal(roc, roc0) and np.array_equal(cor, cor0)
    assert np.array_equal(off, O.exclusive_offsets(O.histogram(idx, 4)))
    out, _ = O.moe_forward_capacity(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], cap)
    out0, _ = O.moe_forward(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"])
    assert np.array_equal(out, out0)


def test_capacity_forward_is_dropless_brute_force_without_dropped_copies():
    """Dropping a copy = giving it gate weight 0 in the dense per-token brute
    force (fp64)."""
    p = _layer(30, 16, 24, 4, 2, seed=42)
    lg = O.gate_logits(p["x"], p["w_gate"])
    idx, g = O.route(lg, None, 2, "softmax")
    cap = O.capacity(30, 4, 2, 0.8)
    roc, _, _, _, dropped = O.permutation_capacity(idx, 4, cap)
    assert dropped > 0
    g0 = np.where(roc.reshape(idx.shape) < 0, 0.0, g)
    ref = O.moe_forward_dense_bruteforce(p["x"], idx, g0, p["w1"], p["w3"], p["w2"])
    out, _ = O.moe_forward_capacity(p["x"], lg, idx, g, p["w1"], p["w3"], p["w2"], cap, dtype=np.float64)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_capacity_backward_finite_differences():
    """Gradients of the layer with drops (routing and the drop pattern held
    fixed) against fp64 central differences: dropped copies have dg = 0 but
    still move the kept copies' renormalised gate weights."""
    n, d, f, e, k = 16, 8, 16, 4, 2
    p = _layer(n, d, f, e, k, "softmax", seed=43, wscale=0.5)
    for key in ("x", "w_gate", "w1", "w3", "w2"):
        p[key] = p[key].astype(np.float64)
    dy = _rng(44).standard_normal((n, d))
    lg = O.gate_logits(p["x"], p["w_gate"], np.float64)
    idx = O.topk_select(O.selection_keys(lg.astype(np.float32), None), k)
    keys = np.sort(O.selection_keys(lg.astype(np.float32), None), axis=1)
    assert (keys[:, -k] - keys[:, -k - 1]).min() > 1e-3
    cap = O.capacity(n, e, k, 0.75)

    def loss_of(pp):
        l2 = O.gate_logits(pp["x"], pp["w_gate"], np.float64)
        g2 = O.gate_weights(l2, idx, "softmax", np.float64)
        o, sv = O.moe_forward_capacity(pp["x"], l2, idx, g2, pp["w1"], pp["w3"], pp["w2"], cap, dtype=np.float64)
        return float((o * dy).sum()), l2, g2, sv

    _, lg, g, saved = loss_of(p)
    assert O.permutation_capacity(idx, e, cap)[4] > 0
    gr = O.moe_backward(dy, p["x"], lg, idx, g, p["w_gate"], p["w1"], p["w3"], p["w2"], saved, "softmax",
                        None, dtype=np.float64)
    r = _rng(45)
    for src, gname in (("x", "dx"), ("w_gate", "dw_gate"), ("w1", "dw1"), ("w2", "dw2")):
        arr = p[src]
        for _ in range(6):
            pos = tuple(int(r.integers(s)) for s in arr.shape)
            old = arr[pos]
            arr[pos] = old + 1e-6
            lp = loss_of(p)[0]
            arr[pos] = old - 1e-6
            lm = loss_of(p)[0]
            arr[pos] = old
            fd = (lp - lm) / 2e-6
            assert abs(fd - gr[gname][pos]) <= 1e-6 * max(1.0, abs(fd)), (gname, pos)


# ------------------------------------------------- FP8 weights, per tile ---
def test_fp8_tile_quantize_scale_and_layout():
    """Per 128 x 128 block: scale = amax / 448, the block maximum encodes to
    +-448, every code is the nearest E4M3 value of w / scale, partial edge
    blocks have their own scale, and a zero block has scale 1."""
    r = _rng(50)
    w = (r.standard_normal((2, 200, 300)) * np.exp2(r.integers(-8, 8, (2, 1, 1)))).astype(np.float32)
    w[1, :128, :128] = 0.0
    codes, scales = O.fp8_tile_quantize(w)
    assert scales.shape == (2, 2, 3) and scales[1, 0, 0] == 1.0
    for e in range(2):
        for i in range(2):
            for j in range(3):
                blk = w[e, 128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]
                cb = codes[e, 128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]
                if not blk.any():
                    assert not cb.any()
                    continue
                sc = np.float32(np.abs(blk).max() / np.float32(448.0))
                assert scales[e, i, j] == sc
                assert np.abs(O.e4m3_decode(cb)).max() == 448.0
                # nearest representable: brute force over the 126 positive values
                grid = np.unique(np.abs(O.e4m3_decode(np.arange(127))))
                v = np.abs(blk.astype(np.float64) / np.float64(sc)).reshape(-1)[:300]
                dist = np.abs(grid[None, :] - v[:, None])
                best = dist.min(axis=1)
                got = np.abs(O.e4m3_decode(cb.reshape(-1)[:300]))
                assert np.allclose(np.abs(got - v), best, rtol=0, atol=1e-12)


def test_fp8_tile_dequantize_round_trip_on_representable_weights():
    """Weights built as E4M3 value x a power-of-two tile scale (bf16 exact)
    come back exactly; a generic weight comes back within E4M3's relative
    step (2^-4 of each element, up to saturation at the block maximum)."""
    r = _rng(51)
    codes = r.integers(0, 127, (130, 260)).astype(np.uint8)
    codes[0, 0] = 0x7E                                   # 448 in every block? one block at least
    vals = O.e4m3_decode(codes) * np.where(r.random((130, 260)) < 0.5, -1, 1)
    w = (vals * 2.0 ** -6).astype(np.float32)            # tile amax -> 448 * 2^-6 only where present
    c2, s2 = O.fp8_tile_quantize(w)
    back = O.fp8_tile_dequantize(c2, s2)
    assert np.allclose(back, O.bf16_round(w), rtol=2 ** -3, atol=0)
    g = r.standard_normal((256, 384)).astype(np.float32)
    c3, s3 = O.fp8_tile_quantize(g)
    b3 = O.fp8_tile_dequantize(c3, s3)
    assert (np.abs(b3 - g) <= np.abs(g) * 2.0 ** -4 + np.repeat(np.repeat(s3, 128, 0), 128, 1) * 2.0 ** -9 + 1e-12).all()


def test_mxfp8_backward_quantises_the_stored_bf16_dyw():
    """What the storage reading changes, worked by hand.  A 32-element row
    of dY with dY[0] = 256 and dY[1] = v = 1.1875 - 2^-20 (fp32), the rest 0,
    on a one-expert, top-1 layer (g = 1, so dYw = dY):

    * block scale: amax 256 = 2^8, exponent floor(log2 256) - 8 = 0, X = 1
      (E8M0 byte 127); 256 -> E4M3 0x78 (exponent field 15, mantissa 0);
    * v lies just below 1.1875, the midpoint of the E4M3 neighbours 1.125
      (0x39: exponent field 7, mantissa 001) and 1.25 (0x3A, mantissa 010),
      so the fp32 operand rounds down to 0x39;
    * bf16(v) = 1.1875 exactly (v is within half a bf16 step, 2^-8, of it),
      a tie, which rounds to the even mantissa 010: 0x3A.

    The oracle's MXFP8 backward quantises dYw as the layer stores it (bf16),
    so the operand of its first quantised GEMM (dh = dYw w2) carries 1.1875
    and code 0x3A; with the identity as storage it carries v and 0x39."""
    v = np.float32(1.1875) - np.float32(2.0 ** -20)
    row = np.zeros((1, 32), np.float32)
    row[0, 0], row[0, 1] = 256.0, v
    codes, scales, _ = O.mx_quantize(row, axis=1)
    assert codes[0, 0] == 0x78 and codes[0, 1] == 0x39 and scales[0, 0] == 127
    stored = O.bf16_round(row)
    assert stored[0, 1] == np.float32(1.1875)
    codes_b, scales_b, _ = O.mx_quantize(stored, axis=1)
    assert codes_b[0, 0] == 0x78 and codes_b[0, 1] == 0x3A and scales_b[0, 0] == 127

    r = _rng(35)
    n, d, f = 1, 32, 32
    x = r.standard_normal((n, d)).astype(np.float32)
    w1, w3 = (r.standard_normal((1, f, d)).astype(np.float32) * np.float32(0.1) for _ in range(2))
    w2 = r.standard_normal((1, d, f)).astype(np.float32) * np.float32(0.1)
    w_gate = r.standard_normal((1, d)).astype(np.float32)
    lg = O.gate_logits(x, w_gate)
    idx, g = O.route(lg, None, 1, "softmax")
    assert g[0, 0] == np.float32(1.0)
    for store, want_val, want_code in ((O.bf16_round, np.float32(1.1875), 0x3A), (lambda a: a, v, 0x39)):
        _, saved = O.moe_forward_mxfp8(x, idx, g, w1, w3, w2, None, return_saved=True, store=store)
        seen = []

        def recording_quant(a, axis):
            seen.append(np.array(a, dtype=np.float64))
            return O.mx_fake_quant(a, axis=axis)
        O.moe_backward_mxfp8(row, x, lg, idx, g, w_gate, w1, w3, w2, saved, "softmax", None,
                             quant=recording_quant, store=store)
        dyw_operand = seen[0]                    # first quantised operand: dYw of dh = dYw w2, along D
        assert dyw_operand.shape == (1, 32) and dyw_operand[0, 1] == want_val
        assert O.mx_quantize(dyw_operand, axis=1)[0][0, 1] == want_code


def test_oracle_pool_runs_the_oracle_unchanged():
    """The parallel runner of the GPU parity tests (spawned processes, expert
    weights shared as bf16 bits) returns what the oracle returns when called
    directly on the same group of tokens."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from oracle_pool import SharedBf16, run_groups
    r = _rng(40)
    n, d, f, e, k = 6, 32, 64, 4, 2
    bf = lambda a: O.bf16_round(a)   # noqa: E731
    x = bf(r.standard_normal((n, d)).astype(np.float32))
    w1, w3 = (bf(r.standard_normal((e, f, d)).astype(np.float32) * np.float32(0.1)) for _ in range(2))
    w2 = bf(r.standard_normal((e, d, f)).astype(np.float32) * np.float32(0.1))
    wg = bf(r.standard_normal((e, d)).astype(np.float32) * np.float32(0.1))
    dy = bf(r.standard_normal((n, d)).astype(np.float32))
    lg = O.gate_logits(x, wg)
    idx, g = O.route(lg, None, k, "softmax")
    bits = lambda a: (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)   # noqa: E731
    shm = {name: SharedBf16(bits(w)) for name, w in (("w1", w1), ("w3", w3), ("w2", w2))}
    try:
        used = np.arange(e)
        job = {"used": used, "w1": shm["w1"].spec, "w3": shm["w3"].spec, "w2": shm["w2"].spec, "x": x,
               "idx": idx, "g": g, "logits": lg, "dy": dy, "w_gate": wg, "shared": None, "gate": "softmax"}
        res = run_groups([dict(job, mxfp8=True), dict(job, mxfp8=False)])
    finally:
        for v in shm.values():
            v.close()
    out_q, saved_q = O.moe_forward_mxfp8(x, idx, g, w1, w3, w2, None, return_saved=True)
    ref_q = O.moe_backward_mxfp8(dy, x, lg, idx, g, wg, w1, w3, w2, saved_q, "softmax", None)
    out, saved = O.moe_forward(x, lg, idx, g, w1, w3, w2, None)
    ref = O.moe_backward(dy, x, lg, idx, g, wg, w1, w3, w2, saved, "softmax", None)
    for got, want_out, want in ((res[0], out_q, ref_q), (res[1], out, ref)):
        np.testing.assert_array_equal(got["out"], want_out)
        for key in ("dx", "dg", "dlogits"):
            np.testing.assert_array_equal(got[key], want[key])
