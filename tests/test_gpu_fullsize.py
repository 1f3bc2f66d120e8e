"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (one MoELayer forward + backward through the C ABI).

The oracle cannot afford the whole batch, so it is compared where it can
compute outputs one by one:

* routing (logits, top-K, histogram, offsets, permutation) on every token;
* layer output, input gradient, gate-weight and router-logit gradients on a
  seeded sample of tokens.  Tokens are independent, so the oracle runs on
  small groups of sampled tokens; inside a group the experts those tokens
  use are re-indexed 0..U-1 (weights, logits columns and gate rows taken in
  the same order), which leaves every compared value unchanged and bounds
  the oracle's memory;
* weight gradients of the most loaded expert: dW_e depends only on the rows
  routed to e, so the oracle runs the K=1 sub-problem made of exactly those
  rows (each with its own gate weight) against expert e alone;
* experts that received no token: weight gradients exactly zero."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import BF16_TOL, np32, rel, routing_agreement
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_dy, make_layer, sample_tokens

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
MX_TOL = 3e-2       # MXFP8 against the quantisation-aware oracle


def _experts(t, used):
    return np.stack([t[int(e)].float().cpu().numpy() for e in used])


@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_full_size_sampled(name):
    cfg = CONFIGS[name]
    torch.cuda.empty_cache()
    p = make_layer(cfg, "cuda")
    dy = make_dy(cfg, "cuda")
    layer = api.MoELayer(cfg, p, train=True)
    out = layer.forward(p["x"])
    gr = layer.backward(dy)
    torch.cuda.synchronize()
    assert layer.device_status()[0] == 0

    x = np32(p["x"])
    wg = np32(p["w_gate"])
    bias = np32(p["bias"])
    # ---- routing on every token
    lg = O.gate_logits(x, wg)
    glg = np32(layer.buf["logits"])
    assert rel(glg, lg) < 1e-5
    keys = O.selection_keys(lg, bias)
    idx, g = O.route(lg, bias, cfg.top_k, cfg.gate)
    gidx = layer.buf["topk_idx"].cpu().numpy()
    tol = 2 * float(np.abs(glg - lg).max()) + 1e-6
    same = routing_agreement(keys, gidx, idx, tol)
    assert same.mean() > 0.999
    gcounts = O.histogram(gidx, cfg.n_exp)
    np.testing.assert_array_equal(layer.buf["counts"].cpu().numpy(), gcounts)
    np.testing.assert_array_equal(layer.buf["offsets"].cpu().numpy(), O.exclusive_offsets(gcounts))
    roc, cor = O.permutation(gidx, cfg.n_exp)
    np.testing.assert_array_equal(layer.buf["row_of_copy"].cpu().numpy(), roc)
    np.testing.assert_array_equal(layer.buf["copy_of_row"].cpu().numpy(), cor)

    shared = (np32(p["ws1"]), np32(p["ws3"]), np32(p["ws2"])) if cfg.n_shared else None
    dyh = np32(dy)

    # ---- per-token outputs and gradients on a token sample, in small groups
    smp = sample_tokens(cfg.n_tok, 48).numpy()
    smp = smp[same[smp]]
    groups, cur, cur_e = [], [], set()
    for t in smp:
        es = set(idx[t].tolist())
        if cur and len(cur_e | es) > 16:
            groups.append(cur)
            cur, cur_e = [], set()
        cur.append(t)
        cur_e |= es
    groups.append(cur)
    got = {k: [] for k in ("out", "dx", "dg", "dlogits")}
    want = {k: [] for k in got}
    for grp in groups:
        grp = np.array(grp)
        used = np.unique(idx[grp])
        ic = np.searchsorted(used, idx[grp]).astype(np.int32)
        lgc = lg[grp][:, used]
        w1, w3, w2 = _experts(p["w1"], used), _experts(p["w3"], used), _experts(p["w2"], used)
        o, saved = O.moe_forward(x[grp], lgc, ic, g[grp], w1, w3, w2, shared)
        rg = O.moe_backward(dyh[grp], x[grp], lgc, ic, g[grp], wg[used], w1, w3, w2, saved, cfg.gate, shared)
        got["out"].append(np32(out)[grp])
        want["out"].append(o)
        got["dx"].append(np32(gr["dx"])[grp])
        want["dx"].append(rg["dx"])
        got["dg"].append(np32(gr["dg"])[grp])
        want["dg"].append(rg["dg"])
        got["dlogits"].append(np32(gr["dlogits"])[grp])
        want["dlogits"].append(np.take_along_axis(rg["dlogits"], ic.astype(np.int64), axis=1))
    # one normwise error over the whole sample (the groups only bound the oracle's memory)
    for key in got:
        assert rel(np.concatenate(got[key]), np.concatenate(want[key])) < BF16_TOL, key

    # ---- weight gradients of the most loaded expert (K=1 sub-problem of its rows)
    counts = O.histogram(idx, cfg.n_exp)
    e_hot = int(np.argmax(counts))
    tok, kk = np.nonzero(idx == e_hot)
    if same[tok].all():
        used = np.array([e_hot])
        w1, w3, w2 = _experts(p["w1"], used), _experts(p["w3"], used), _experts(p["w2"], used)
        i1 = np.zeros((len(tok), 1), np.int32)
        g1 = g[tok, kk][:, None]
        lg1 = lg[tok][:, [e_hot]]
        o, saved = O.moe_forward(x[tok], lg1, i1, g1, w1, w3, w2, None)
        rg = O.moe_backward(dyh[tok], x[tok], lg1, i1, g1, wg[used], w1, w3, w2, saved, cfg.gate, None)
        for key in ("dw1", "dw3", "dw2"):
            assert rel(gr[key][e_hot].cpu().numpy(), rg[key][0]) < BF16_TOL, key
    for e in np.nonzero(gcounts == 0)[0][:2]:
        assert not gr["dw1"][int(e)].any() and not gr["dw2"][int(e)].any()
    del layer, p
    torch.cuda.empty_cache()


def test_full_size_sampled_mxfp8_dsv3():
    """The DeepSeek-V3-shaped layer with MXFP8 expert GEMMs, forward and
    backward at full size, against the quantisation-aware oracle.  Row-wise
    quantisation (x, h along D/F; dYw, da1, da3 along D/F) keeps token rows
    independent, so outputs and input-side gradients are checked on a token
    sample; the weight gradients of the most loaded expert depend on its
    tokens in 32-row blocks, so the oracle runs that expert's whole row set."""
    cfg = CONFIGS["dsv3"].replace(precision="mxfp8")
    torch.cuda.empty_cache()
    p = make_layer(cfg, "cuda")
    dy = make_dy(cfg, "cuda")
    layer = api.MoELayer(cfg, p, train=True)
    out = layer.forward(p["x"])
    gr = layer.backward(dy)
    torch.cuda.synchronize()
    assert layer.device_status()[0] == 0

    x = np32(p["x"])
    wg = np32(p["w_gate"])
    bias = np32(p["bias"])
    lg = O.gate_logits(x, wg)
    glg = np32(layer.buf["logits"])
    keys = O.selection_keys(lg, bias)
    idx, g = O.route(lg, bias, cfg.top_k, cfg.gate)
    gidx = layer.buf["topk_idx"].cpu().numpy()
    tol = 2 * float(np.abs(glg - lg).max()) + 1e-6
    same = routing_agreement(keys, gidx, idx, tol)
    shared = (np32(p["ws1"]), np32(p["ws3"]), np32(p["ws2"]))
    dyh = np32(dy)

    # a token sample whose experts stay within 16 (every expert's weights are
    # quantised once per contraction axis by the oracle, which bounds its time)
    cand = sample_tokens(cfg.n_tok, 512).numpy()
    grp, used_e = [], set()
    for t in cand:
        es = set(idx[t].tolist())
        if same[t] and len(used_e | es) <= 16:
            grp.append(t)
            used_e |= es
        if len(grp) == 8:
            break
    grp = np.array(grp)
    assert len(grp) >= 2
    used = np.unique(idx[grp])
    ic = np.searchsorted(used, idx[grp]).astype(np.int32)
    lgc = lg[grp][:, used]
    w1, w3, w2 = _experts(p["w1"], used), _experts(p["w3"], used), _experts(p["w2"], used)
    o, saved = O.moe_forward_mxfp8(x[grp], ic, g[grp], w1, w3, w2, shared, return_saved=True)
    rg = O.moe_backward_mxfp8(dyh[grp], x[grp], lgc, ic, g[grp], wg[used], w1, w3, w2, saved, cfg.gate, shared)
    assert rel(np32(out)[grp], o) < MX_TOL, "out"
    assert rel(np32(gr["dx"])[grp], rg["dx"]) < MX_TOL, "dx"
    assert rel(np32(gr["dg"])[grp], rg["dg"]) < MX_TOL, "dg"
    assert rel(np32(gr["dlogits"])[grp], np.take_along_axis(rg["dlogits"], ic.astype(np.int64), axis=1)) < MX_TOL

    counts = O.histogram(idx, cfg.n_exp)
    e_hot = int(np.argmax(counts))
    tok, kk = np.nonzero(idx == e_hot)
    if same[tok].all():
        used = np.array([e_hot])
        w1, w3, w2 = _experts(p["w1"], used), _experts(p["w3"], used), _experts(p["w2"], used)
        i1 = np.zeros((len(tok), 1), np.int32)
        g1 = g[tok, kk][:, None]
        lg1 = lg[tok][:, [e_hot]]
        _, saved = O.moe_forward_mxfp8(x[tok], i1, g1, w1, w3, w2, None, return_saved=True)
        rg = O.moe_backward_mxfp8(dyh[tok], x[tok], lg1, i1, g1, wg[used], w1, w3, w2, saved, cfg.gate, None)
        for key in ("dw1", "dw3", "dw2"):
            assert rel(gr[key][e_hot].cpu().numpy(), rg[key][0]) < MX_TOL, key
    for e in np.nonzero(O.histogram(gidx, cfg.n_exp) == 0)[0][:2]:
        assert not gr["dw1"][int(e)].any() and not gr["dw2"][int(e)].any()
    del layer, p
    torch.cuda.empty_cache()
