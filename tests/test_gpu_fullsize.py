"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (one MoELayer forward + backward through the C ABI).

The oracle cannot afford the whole batch, so it is compared where it can
compute outputs one by one:

* routing (logits, top-K, histogram, offsets, permutation) on every token;
* layer output, input gradient, gate-weight and router-logit gradients on a
  seeded sample of tokens, as one normwise error over the sample and per
  token (99th percentile within twice the tolerance).  Tokens are independent, so the oracle runs on
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
from oracle_pool import SharedBf16, run_groups, token_groups
from parity_util import BF16_TOL, check_rows, np32, rel, routing_agreement
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_dy, make_layer, sample_tokens, skewed_logits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
MX_TOL = 3e-2       # MXFP8 against the quantisation-aware oracle


_check_sample = check_rows


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
    # one normwise error over the whole sample (the groups only bound the oracle's memory), and per token
    for key in got:
        _check_sample(np.concatenate(got[key]), np.concatenate(want[key]), BF16_TOL, key)

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


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _jobs(shm, x, dy, lg, idx, g, groups, wg, gate, shared, mxfp8=True):
    jobs = []
    for grp in groups:
        used = np.unique(idx[grp])
        jobs.append({"used": used, "w1": shm["w1"].spec, "w3": shm["w3"].spec, "w2": shm["w2"].spec,
                     "x": x[grp], "idx": np.searchsorted(used, idx[grp]).astype(np.int32), "g": g[grp],
                     "logits": lg[grp][:, used], "dy": dy[grp], "w_gate": wg[used], "shared": shared,
                     "gate": gate, "mxfp8": mxfp8})
    return jobs


def _expert_job(shm, x, dy, lg, idx, g, e, wg, gate, mxfp8=True):
    """The K=1 sub-problem of expert e: exactly its rows (ascending token
    order, each with its own gate weight), against expert e alone.  dW_e
    depends only on these rows (MXFP8: quantised in 32-row blocks from the
    expert's first row, as in the whole layer)."""
    tok, kk = np.nonzero(idx == e)
    used = np.array([e])
    return {"used": used, "w1": shm["w1"].spec, "w3": shm["w3"].spec, "w2": shm["w2"].spec, "x": x[tok],
            "idx": np.zeros((len(tok), 1), np.int32), "g": g[tok, kk][:, None], "logits": lg[tok][:, [e]],
            "dy": dy[tok], "w_gate": wg[used], "shared": None, "gate": gate, "mxfp8": mxfp8,
            "keep": ("dw1", "dw3", "dw2")}, tok


def _mx_layer_run(cfg, p, dy, logits=None):
    """One MXFP8 layer forward + backward on the GPU (routing by the layer's
    own gate and bias, or from the given fp32 logits with a zero bias), with
    the outputs the checks need copied to the host."""
    layer = api.MoELayer(cfg, p, train=True)
    b = layer.buf
    if logits is None:
        out = layer.forward(p["x"])
    else:
        zero = torch.zeros(cfg.n_exp, dtype=torch.float32, device="cuda")
        api.moe_route_from_logits(layer.desc, logits, zero, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                                  layer.ws)
        b["logits"].copy_(logits)
        layer.x = p["x"]
        out = layer._forward_mx(p["x"])
    gr = layer.backward(dy)
    torch.cuda.synchronize()
    assert layer.device_status()[0] == 0
    res = {"out": np32(out), "dx": np32(gr["dx"]), "dg": np32(gr["dg"]), "dlogits": np32(gr["dlogits"]),
           "idx": b["topk_idx"].cpu().numpy(), "topk_w": np32(b["topk_w"]), "logits": np32(b["logits"]),
           "counts": b["counts"].cpu().numpy(), "dw": {}}
    return layer, gr, res


def _compare_groups(res, groups, results, tol):
    got = {k: [] for k in ("out", "dx", "dg", "dlogits")}
    want = {k: [] for k in got}
    for grp, rg in zip(groups, results):
        used = np.unique(res["oracle_idx"][grp])
        ic = np.searchsorted(used, res["oracle_idx"][grp]).astype(np.int64)
        for key in ("out", "dx", "dg"):
            got[key].append(res[key][grp])
            want[key].append(rg[key])
        got["dlogits"].append(res["dlogits"][grp])
        want["dlogits"].append(np.take_along_axis(rg["dlogits"], ic, axis=1))
    for key in got:
        _check_sample(np.concatenate(got[key]), np.concatenate(want[key]), tol, key)


def test_full_size_sampled_mxfp8_dsv3():
    """The DeepSeek-V3-shaped layer with MXFP8 expert GEMMs, forward and
    backward at full size, against the quantisation-aware oracle.  Row-wise
    quantisation (x, h along D/F; dYw, da1, da3 along D/F) keeps token rows
    independent, so outputs and input-side gradients are checked on a sample
    of 32 tokens (groups with few experts, run by the oracle in parallel
    processes); the weight gradients of the most loaded expert depend on its
    tokens in 32-row blocks, so the oracle runs that expert's whole row set."""
    cfg = CONFIGS["dsv3"].replace(precision="mxfp8")
    torch.cuda.empty_cache()
    p = make_layer(cfg, "cuda")
    dy = make_dy(cfg, "cuda")
    layer, gr, res = _mx_layer_run(cfg, p, dy)
    x, wg, bias, dyh = np32(p["x"]), np32(p["w_gate"]), np32(p["bias"]), np32(dy)
    lg = O.gate_logits(x, wg)
    keys = O.selection_keys(lg, bias)
    idx, g = O.route(lg, bias, cfg.top_k, cfg.gate)
    tol = 2 * float(np.abs(res["logits"] - lg).max()) + 1e-6
    same = routing_agreement(keys, res["idx"], idx, tol)
    res["oracle_idx"] = idx
    shared = (np32(p["ws1"]), np32(p["ws3"]), np32(p["ws2"]))
    cand = [t for t in sample_tokens(cfg.n_tok, 1024).numpy() if same[t]]
    groups = token_groups(idx, cand, max_experts=16, max_tokens=32)
    assert sum(len(x_) for x_ in groups) == 32
    e_hot = int(np.argmax(O.histogram(idx, cfg.n_exp)))
    hot_ok = bool(same[np.nonzero(idx == e_hot)[0]].all())
    hot_dw = {k: gr[k][e_hot].cpu().numpy() for k in ("dw1", "dw3", "dw2")}
    empty = [int(e) for e in np.nonzero(res["counts"] == 0)[0][:2]]
    empty_ok = all(not gr["dw1"][e].any() and not gr["dw2"][e].any() for e in empty)
    shm = {k: SharedBf16(_bits(p[k])) for k in ("w1", "w3", "w2")}
    del layer, gr, p
    torch.cuda.empty_cache()
    try:
        jobs = _jobs(shm, x, dyh, lg, idx, g, groups, wg, cfg.gate, shared)
        hot_job, _ = _expert_job(shm, x, dyh, lg, idx, g, e_hot, wg, cfg.gate)
        results = run_groups(jobs + ([hot_job] if hot_ok else []))
    finally:
        for v in shm.values():
            v.close()
    _compare_groups(res, groups, results[:len(groups)], MX_TOL)
    if hot_ok:
        for key in ("dw1", "dw3", "dw2"):
            assert rel(hot_dw[key], results[-1][key][0]) < MX_TOL, key
    assert empty_ok


def test_full_size_sampled_mxfp8_mixtral(monkeypatch):
    """The Mixtral-shaped layer with MXFP8 expert GEMMs (~1024 rows per
    expert, contractions of 4096 and 14336), forward and backward at full
    size, in both GEMM forms (one-SM and CTA pair), against the same
    quantisation-aware oracle results: a sample of 32 tokens, and the
    weight gradients of the most loaded expert over its whole row set."""
    cfg = CONFIGS["mixtral"].replace(precision="mxfp8")
    torch.cuda.empty_cache()
    p = make_layer(cfg, "cuda")
    dy = make_dy(cfg, "cuda")
    x, wg, dyh = np32(p["x"]), np32(p["w_gate"]), np32(dy)
    lg = O.gate_logits(x, wg)
    keys = O.selection_keys(lg, None)
    idx, g = O.route(lg, None, cfg.top_k, cfg.gate)
    e_hot = int(np.argmax(O.histogram(idx, cfg.n_exp)))
    runs = {}
    for form in ("0", "1"):
        monkeypatch.setenv("MOE_GEMM_CTA_PAIR", form)
        layer, gr, res = _mx_layer_run(cfg, p, dy)
        tol = 2 * float(np.abs(res["logits"] - lg).max()) + 1e-6
        res["same"] = routing_agreement(keys, res["idx"], idx, tol)
        res["oracle_idx"] = idx
        res["hot_dw"] = {k: gr[k][e_hot].cpu().numpy() for k in ("dw1", "dw3", "dw2")}
        runs[form] = res
        del layer, gr
        torch.cuda.empty_cache()
    same = runs["0"]["same"] & runs["1"]["same"]
    cand = [t for t in sample_tokens(cfg.n_tok, 1024).numpy() if same[t]]
    groups = token_groups(idx, cand, max_experts=4, max_tokens=32)
    assert sum(len(x_) for x_ in groups) == 32
    hot_ok = bool(same[np.nonzero(idx == e_hot)[0]].all())
    shm = {k: SharedBf16(_bits(p[k])) for k in ("w1", "w3", "w2")}
    del p
    torch.cuda.empty_cache()
    try:
        jobs = _jobs(shm, x, dyh, lg, idx, g, groups, wg, cfg.gate, None)
        hot_job, _ = _expert_job(shm, x, dyh, lg, idx, g, e_hot, wg, cfg.gate)
        results = run_groups(jobs + ([hot_job] if hot_ok else []))
    finally:
        for v in shm.values():
            v.close()
    for form, res in runs.items():
        _compare_groups(res, groups, results[:len(groups)], MX_TOL)
        if hot_ok:
            for key in ("dw1", "dw3", "dw2"):
                assert rel(res["hot_dw"][key], results[-1][key][0]) < MX_TOL, (form, key)


@pytest.mark.parametrize("skew", ["uniform", "zipf", "half0"])
def test_full_size_mxfp8_dsv3_load_skews(skew):
    """The MXFP8 layer (DeepSeek-V3 shapes) forward and backward under the
    load skews of the MXFP8 configuration: i.i.d. logits (near-uniform
    loads), Zipf(s=1) expert preference (heavy experts saturate at one copy
    per token), and half of the tokens on expert 0 (2048 rows, 16x the
    mean).  Routing comes from the same fp32 logits on both sides (bit for
    bit); outputs and input-side gradients are compared on a token sample,
    and the weight gradients of the most loaded expert (expert 0 under the
    half-on-one skew) in full, against the quantisation-aware oracle."""
    cfg = CONFIGS["dsv3"].replace(precision="mxfp8")
    torch.cuda.empty_cache()
    p = make_layer(cfg, "cuda")
    dy = make_dy(cfg, "cuda")
    lg = skewed_logits(cfg.n_tok, cfg.n_exp, skew)
    layer, gr, res = _mx_layer_run(cfg, p, dy, logits=lg.cuda())
    lgh = lg.numpy()
    idx, g = O.route(lgh, np.zeros(cfg.n_exp, np.float32), cfg.top_k, cfg.gate)
    np.testing.assert_array_equal(res["idx"], idx)
    np.testing.assert_array_equal(res["counts"], O.histogram(idx, cfg.n_exp))
    res["oracle_idx"] = idx
    counts = O.histogram(idx, cfg.n_exp)
    e_hot = int(np.argmax(counts))
    if skew == "half0":
        assert e_hot == 0 and counts[0] >= cfg.n_tok // 2
    x, wg, dyh = np32(p["x"]), np32(p["w_gate"]), np32(dy)
    shared = (np32(p["ws1"]), np32(p["ws3"]), np32(p["ws2"]))
    groups = token_groups(idx, sample_tokens(cfg.n_tok, 512).numpy(), max_experts=16, max_tokens=8)
    hot_dw = {k: gr[k][e_hot].cpu().numpy() for k in ("dw1", "dw3", "dw2")}
    shm = {k: SharedBf16(_bits(p[k])) for k in ("w1", "w3", "w2")}
    del layer, gr, p
    torch.cuda.empty_cache()
    try:
        jobs = _jobs(shm, x, dyh, lgh, idx, g, groups, wg, cfg.gate, shared)
        hot_job, _ = _expert_job(shm, x, dyh, lgh, idx, g, e_hot, wg, cfg.gate)
        results = run_groups(jobs + [hot_job])
    finally:
        for v in shm.values():
            v.close()
    _compare_groups(res, groups, results[:-1], MX_TOL)
    for key in ("dw1", "dw3", "dw2"):
        assert rel(hot_dw[key], results[-1][key][0]) < MX_TOL, key
