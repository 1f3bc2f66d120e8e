"""GPU parity: every entry point of the C ABI against the CPU oracle on the
same seeded inputs.  Integer outputs (routing, histogram, offsets,
permutation, bias update) are compared bit for bit; floating-point outputs
by normwise relative error (bf16 storage, fp32 accumulation: 5e-3)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import BF16_TOL, check_rows, host_params, np32, rel, routing_agreement, to_dev
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, MoEConfig, make_dy, make_layer, route_bias, skewed_logits

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "small_softmax", "small_sigmoid", "small_fine"]


def _i32(*s):
    return torch.empty(s, dtype=torch.int32, device="cuda")


def _f32(*s):
    return torch.empty(s, dtype=torch.float32, device="cuda")


def _bf(*s):
    return torch.empty(s, dtype=torch.bfloat16, device="cuda")


def _ws(cfg):
    d = api.make_desc(cfg)
    _, b = api.moe_workspace_size(d)
    ws = torch.empty(b, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    return d, ws


def _status_ok(ws):
    bits, site = api.moe_get_device_status(ws)
    assert bits == 0, f"device status {bits} (site {site})"


@pytest.fixture(params=["1", "0"], ids=["cta_pair", "one_sm"])
def gemm_form(request, monkeypatch):
    """Runs a test with the grouped GEMMs forced to the 2-SM (CTA pair) form
    or to the one-SM form; by default the library picks the form from the
    group sizes."""
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", request.param)
    return request.param


def _layer(name):
    cfg = CONFIGS[name] if isinstance(name, str) else name
    p_cpu = make_layer(cfg, "cpu")
    return cfg, to_dev(p_cpu), host_params(p_cpu)


def _shared(h):
    return (h["ws1"], h["ws3"], h["ws2"]) if "ws1" in h else None


# ------------------------------------------------------------- routing
@pytest.mark.parametrize("name,mode", [("tiny", "uniform"), ("tiny", "ties"), ("small_fine", "zipf"),
                                       ("small_fine", "half0"), ("small_sigmoid", "ties"),
                                       ("dsv3", "uniform"), ("dsv3", "zipf"), ("dsv3", "half0"),
                                       ("dsv3", "ties"), ("mixtral", "uniform")])
def test_route_from_logits_bitexact(name, mode):
    cfg = CONFIGS[name]
    n, e, k = cfg.n_tok, cfg.n_exp, cfg.top_k
    lg = skewed_logits(n, e, mode)
    lg[:3] = -0.0 if mode == "ties" else lg[:3]
    bias = route_bias(cfg)
    d, ws = _ws(cfg)
    idx, w, cnt, off = _i32(n, k), _f32(n, k), _i32(e), _i32(e + 1)
    api.moe_route_from_logits(d, lg.cuda(), None if bias is None else bias.cuda(), idx, w, cnt, off, ws)
    _status_ok(ws)
    lgh = lg.numpy()
    bh = None if bias is None else bias.numpy()
    ridx, rw = O.route(lgh, bh, k, cfg.gate)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=1e-6)
    counts = O.histogram(ridx, e)
    np.testing.assert_array_equal(cnt.cpu().numpy(), counts)
    np.testing.assert_array_equal(off.cpu().numpy(), O.exclusive_offsets(counts))


@pytest.mark.parametrize("e,k,mode", [(1024, 32, "uniform"), (1024, 32, "ties"), (1000, 7, "zipf")])
def test_route_from_logits_widest(e, k, mode):
    """The most experts (1024: 32 per lane) and the largest K the selection
    takes (32: every lane holds a pick), and E off a multiple of 32."""
    n = 333
    cfg = MoEConfig("widest", n, 64, 64, e, k)
    lg = skewed_logits(n, e, mode)
    d, ws = _ws(cfg)
    idx, w, cnt, off = _i32(n, k), _f32(n, k), _i32(e), _i32(e + 1)
    api.moe_route_from_logits(d, lg.cuda(), None, idx, w, cnt, off, ws)
    _status_ok(ws)
    ridx, rw = O.route(lg.numpy(), None, k, cfg.gate)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=1e-6)
    counts = O.histogram(ridx, e)
    np.testing.assert_array_equal(cnt.cpu().numpy(), counts)
    np.testing.assert_array_equal(off.cpu().numpy(), O.exclusive_offsets(counts))


# extra router shapes: E = 24 and 32 (fused router with 3 and 4 column
# tiles of 8 experts, token counts off the 16-token tile), a bias; E > 32
# through the logits GEMM and the one-kernel tail: 79 token tiles fill the
# GPU, so no contraction slices (the tail reads the logits themselves), and
# 45 token tiles with six k-blocks, so three slices (E = 96: lanes past E)
ROUTER_EXTRA = {
    "router_e24": MoEConfig("router_e24", 515, 128, 64, 24, 3),
    "router_e32": MoEConfig("router_e32", 1001, 192, 64, 32, 4, gate="sigmoid", use_bias=True, bias_beta=0.5,
                            n_cold=2),
    "router_e64_noslice": MoEConfig("router_e64_noslice", 10000, 64, 64, 64, 6),
    "router_e96_3slices": MoEConfig("router_e96_3slices", 5760, 384, 64, 96, 4, gate="sigmoid"),
    # the widest router: 1024 experts (four 256-column tiles of the logits GEMM), top-32
    "router_e1024": MoEConfig("router_e1024", 700, 128, 64, 1024, 32),
}


@pytest.mark.parametrize("name", SMALL + ["dsv3"] + list(ROUTER_EXTRA))
def test_route_gate_gemm(name):
    cfg = ROUTER_EXTRA.get(name) or CONFIGS[name]
    p_cpu = make_layer(cfg.replace(d_ff=64), "cpu") if name == "dsv3" else make_layer(cfg, "cpu")
    x, wg = p_cpu["x"], p_cpu["w_gate"]
    bias = p_cpu["bias"]
    n, e, k = cfg.n_tok, cfg.n_exp, cfg.top_k
    d, ws = _ws(cfg)
    lg, idx, w, cnt, off = _f32(n, e), _i32(n, k), _f32(n, k), _i32(e), _i32(e + 1)
    api.moe_route(d, x.cuda(), wg.cuda(), None if bias is None else bias.cuda(), lg, idx, w, cnt, off, ws)
    _status_ok(ws)
    ref_lg = O.gate_logits(np32(x), np32(wg))
    glg = lg.cpu().numpy()
    assert rel(glg, ref_lg) < 1e-5
    bh = None if bias is None else bias.numpy()
    keys = O.selection_keys(ref_lg, bh)
    ridx, rw = O.route(ref_lg, bh, k, cfg.gate)
    tol = 2 * float(np.abs(glg - ref_lg).max()) + 1e-6
    same = routing_agreement(keys, idx.cpu().numpy(), ridx, tol)
    assert same.mean() > 0.99
    np.testing.assert_allclose(w.cpu().numpy()[same], rw[same], rtol=0, atol=2e-5)
    # the device histogram and offsets are exactly those of the device's own routing
    gidx = idx.cpu().numpy()
    np.testing.assert_array_equal(cnt.cpu().numpy(), O.histogram(gidx, e))
    np.testing.assert_array_equal(off.cpu().numpy(), O.exclusive_offsets(O.histogram(gidx, e)))


# ------------------------------------------------------------- permutation
# more than 65536 copies: the token-chunked map kernels (three launches)
# instead of the single-CTA pass
LARGE_R = MoEConfig("large_r", 9000, 64, 64, 16, 8)


@pytest.mark.parametrize("name", SMALL + ["dsv3", "large_r"])
def test_permute_bitexact(name):
    cfg = LARGE_R if name == "large_r" else CONFIGS[name]
    n, dm, e, k = cfg.n_tok, cfg.d_model, cfg.n_exp, cfg.top_k
    lg = skewed_logits(n, e, "zipf" if e > 8 else "uniform").numpy()
    ridx, _ = O.route(lg, None, k, cfg.gate)
    off = O.exclusive_offsets(O.histogram(ridx, e))
    x = make_layer(cfg.replace(d_ff=64, n_exp=1, top_k=1, use_bias=False, n_shared=0), "cpu")["x"]
    d, ws = _ws(cfg)
    roc, cor, xp = _i32(n * k), _i32(n * k), _bf(n * k, dm)
    api.moe_permute(d, x.cuda(), torch.from_numpy(ridx).cuda(), torch.from_numpy(off).cuda(), roc, cor, xp, ws)
    _status_ok(ws)
    rroc, rcor = O.permutation(ridx, e)
    np.testing.assert_array_equal(roc.cpu().numpy(), rroc)
    np.testing.assert_array_equal(cor.cpu().numpy(), rcor)
    xb = x.view(torch.int16).numpy()
    np.testing.assert_array_equal(xp.cpu().view(torch.int16).numpy(), xb[rcor // k])
    # the maps alone (one-CTA form up to 65536 copies, token-chunked beyond): the same maps
    roc2, cor2 = _i32(n * k), _i32(n * k)
    api.moe_permute_maps(d, torch.from_numpy(ridx).cuda(), torch.from_numpy(off).cuda(), roc2, cor2, ws)
    _status_ok(ws)
    np.testing.assert_array_equal(roc2.cpu().numpy(), rroc)
    np.testing.assert_array_equal(cor2.cpu().numpy(), rcor)


def test_permute_twice_in_a_row_and_after_other_sizes():
    """The single-pass permute keeps a chunk ticket and a generation counter
    in the workspace between calls: repeated calls, and calls of another
    size on the same workspace, give the same maps and rows."""
    cfg = CONFIGS["small_fine"]
    n, dm, e, k = cfg.n_tok, cfg.d_model, cfg.n_exp, cfg.top_k
    d, ws = _ws(cfg)
    x = make_layer(cfg.replace(d_ff=64, n_exp=1, top_k=1, use_bias=False, n_shared=0), "cpu")["x"].cuda()
    for rep, ntok in enumerate((n, n, 100, n)):
        c = cfg.replace(n_tok=ntok)
        lg = skewed_logits(ntok, e, "zipf", seed=20 + rep).numpy()
        ridx, _ = O.route(lg, None, k, c.gate)
        off = O.exclusive_offsets(O.histogram(ridx, e))
        dd = api.make_desc(c)
        roc, cor, xp = _i32(ntok * k), _i32(ntok * k), _bf(ntok * k, dm)
        api.moe_permute(dd, x[:ntok].contiguous(), torch.from_numpy(ridx).cuda(), torch.from_numpy(off).cuda(), roc,
                        cor, xp, ws)
        _status_ok(ws)
        rroc, rcor = O.permutation(ridx, e)
        np.testing.assert_array_equal(roc.cpu().numpy(), rroc)
        np.testing.assert_array_equal(cor.cpu().numpy(), rcor)
        np.testing.assert_array_equal(xp.cpu().view(torch.int16).numpy(),
                                      x[:ntok].cpu().view(torch.int16).numpy()[rcor // k])


# ------------------------------------------------------------- routing and permute in one launch
# E <= 32 layers; LARGE_E8: more 16-token tiles (563) than resident CTAs, so
# every CTA routes and copies several tiles on either side of the barrier
LARGE_E8 = MoEConfig("large_e8", 9000, 128, 64, 8, 2)
FUSED = ["tiny", "small_softmax", "small_sigmoid", "router_e24", "router_e32", "large_e8",
         "single_token", "one_expert", "k_equals_e", "hot_expert"]


@pytest.mark.parametrize("name", FUSED)
def test_route_permute_equals_route_then_permute(name):
    """moe_route_permute gives, bit for bit, what moe_route followed by
    moe_permute give (every output), twice in a row on one workspace (the
    grid barrier's words are reused), and its maps are the oracle's stable
    permutation of its own routing."""
    cfg = ({"large_e8": LARGE_E8}.get(name) or ROUTER_EXTRA.get(name) or {c.name: c for c in EDGE}.get(name)
           or CONFIGS[name])
    p_cpu = make_layer(cfg.replace(d_ff=64), "cpu")
    x, wg, bias = p_cpu["x"].cuda(), p_cpu["w_gate"].cuda(), p_cpu["bias"]
    bias = None if bias is None else bias.cuda()
    n, dm, e, k = cfg.n_tok, cfg.d_model, cfg.n_exp, cfg.top_k
    r = n * k
    d, ws = _ws(cfg)

    def outs():
        return dict(lg=_f32(n, e), idx=_i32(n, k), w=_f32(n, k), cnt=_i32(e), off=_i32(e + 1), roc=_i32(r),
                    cor=_i32(r), xp=_bf(r, dm))

    a = outs()
    api.moe_route(d, x, wg, bias, a["lg"], a["idx"], a["w"], a["cnt"], a["off"], ws)
    api.moe_permute(d, x, a["idx"], a["off"], a["roc"], a["cor"], a["xp"], ws)
    _status_ok(ws)
    for rep in range(2):
        b = outs()
        api.moe_route_permute(d, x, wg, bias, b["lg"], b["idx"], b["w"], b["cnt"], b["off"], b["roc"], b["cor"],
                              b["xp"], ws)
        _status_ok(ws)
        for key in a:
            ga, gb = a[key].cpu(), b[key].cpu()
            if ga.dtype == torch.bfloat16:
                ga, gb = ga.view(torch.int16), gb.view(torch.int16)
            elif ga.dtype == torch.float32:
                ga, gb = ga.view(torch.int32), gb.view(torch.int32)
            assert torch.equal(ga, gb), (key, rep)
    rroc, rcor = O.permutation(b["idx"].cpu().numpy(), e)
    np.testing.assert_array_equal(b["roc"].cpu().numpy(), rroc)
    np.testing.assert_array_equal(b["cor"].cpu().numpy(), rcor)


def test_route_permute_rejects_what_it_does_not_cover():
    """More than 32 experts or MXFP8 rows: an argument error, nothing launched."""
    for cfg in (CONFIGS["small_fine"], CONFIGS["small_softmax"].replace(precision="mxfp8")):
        n, dm, e, k = cfg.n_tok, cfg.d_model, cfg.n_exp, cfg.top_k
        d, ws = _ws(cfg)
        with pytest.raises(api.MoEError):
            api.moe_route_permute(d, _bf(n, dm), _bf(e, dm), None, _f32(n, e), _i32(n, k), _f32(n, k), _i32(e),
                                  _i32(e + 1), _i32(n * k), _i32(n * k), _bf(n * k, dm), ws)
        _status_ok(ws)


# ------------------------------------------------------------- grouped FFN
def _oracle_route(cfg, h):
    lg = O.gate_logits(h["x"], h["w_gate"])
    idx, g = O.route(lg, h.get("bias"), cfg.top_k, cfg.gate)
    return lg, idx, g


@pytest.mark.parametrize("name", SMALL)
def test_grouped_ffn(name, gemm_form):
    cfg, p, h = _layer(name)
    n, dm, f, e, k = cfg.n_tok, cfg.d_model, cfg.d_ff, cfg.n_exp, cfg.top_k
    r, fs = cfg.rows, cfg.d_ff_shared
    lg, idx, g = _oracle_route(cfg, h)
    off = O.exclusive_offsets(O.histogram(idx, e))
    _, cor = O.permutation(idx, e)
    xperm = p["x"][torch.from_numpy(cor // k).long().cuda()].contiguous()
    d, ws = _ws(cfg)
    a1, a3, hh, yp = _bf(r, f), _bf(r, f), _bf(r, f), _bf(r, dm)
    sh = cfg.n_shared
    a1s, a3s, hs, ys = (_bf(n, fs), _bf(n, fs), _bf(n, fs), _bf(n, dm)) if sh else (None,) * 4
    api.moe_grouped_ffn(d, xperm, torch.from_numpy(off).cuda(), p["x"], p["w1"], p["w3"], p["w2"], p.get("ws1"),
                        p.get("ws3"), p.get("ws2"), a1, a3, hh, a1s, a3s, hs, yp, ys, ws)
    _status_ok(ws)
    xph = h["x"][cor // k]
    ref_y = np.empty((r, dm), np.float32)
    ref_a1 = np.empty((r, f), np.float32)
    ref_h = np.empty((r, f), np.float32)
    for ex in range(e):
        rows = slice(off[ex], off[ex + 1])
        if off[ex] == off[ex + 1]:
            continue
        y, ra1, ra3, rh = O.swiglu_expert(xph[rows], h["w1"][ex], h["w3"][ex], h["w2"][ex])
        ref_y[rows], ref_a1[rows], ref_h[rows] = y, ra1, rh
    assert rel(np32(a1), ref_a1) < BF16_TOL
    assert rel(np32(hh), ref_h) < BF16_TOL
    assert rel(np32(yp), ref_y) < BF16_TOL
    if sh:
        y, _, _, rh = O.swiglu_expert(h["x"], h["ws1"], h["ws3"], h["ws2"])
        assert rel(np32(hs), rh) < BF16_TOL
        assert rel(np32(ys), y) < BF16_TOL


@pytest.mark.parametrize("name", SMALL)
def test_combine(name):
    cfg = CONFIGS[name]
    n, dm, k = cfg.n_tok, cfg.d_model, cfg.top_k
    gen = torch.Generator().manual_seed(5)
    yp = torch.randn(n * k, dm, generator=gen).to(torch.bfloat16)
    ys = torch.randn(n, dm, generator=gen).to(torch.bfloat16) if cfg.n_shared else None
    w = torch.rand(n, k, generator=gen)
    roc = torch.randperm(n * k, generator=gen).to(torch.int32)
    d, _ = _ws(cfg)
    out = _bf(n, dm)
    api.moe_combine(d, yp.cuda(), roc.cuda(), w.cuda(), None if ys is None else ys.cuda(), out)
    torch.cuda.synchronize()
    ref = (w.double()[:, :, None] * yp.double()[roc.long()].view(n, k, dm)).sum(1)
    if ys is not None:
        ref += ys.double()
    assert rel(np32(out), ref.numpy()) < 4e-3   # bf16 rounding of the output only


# ------------------------------------------------------------- whole layer
def _run_layer(cfg, p, dy=None):
    layer = api.MoELayer(cfg, p, train=dy is not None)
    out = layer.forward(p["x"])
    grads = layer.backward(dy) if dy is not None else None
    torch.cuda.synchronize()
    bits, site = layer.device_status()
    assert bits == 0, f"device status {bits} (site {site})"
    return layer, out, grads


@pytest.mark.parametrize("name", SMALL)
def test_forward_end_to_end(name):
    cfg, p, h = _layer(name)
    layer, out, _ = _run_layer(cfg, p)
    lg, idx, g = _oracle_route(cfg, h)
    keys = O.selection_keys(lg, h.get("bias"))
    tol = 2 * float(np.abs(np32(layer.buf["logits"]) - lg).max()) + 1e-6
    same = routing_agreement(keys, layer.buf["topk_idx"].cpu().numpy(), idx, tol)
    ref, _ = O.moe_forward(h["x"], lg, idx, g, h["w1"], h["w3"], h["w2"], _shared(h))
    check_rows(np32(out)[same], ref[same], BF16_TOL, "out")


def _expert_mask(idx_gpu, idx_ref, same, e):
    """Experts whose token sets agree on both sides (their weight gradients are comparable)."""
    bad = set(np.unique(idx_gpu[~same]).tolist()) | set(np.unique(idx_ref[~same]).tolist())
    return np.array([ex not in bad for ex in range(e)])


@pytest.mark.parametrize("name", SMALL)
def test_backward_end_to_end(name, gemm_form):
    cfg, p, h = _layer(name)
    dy = make_dy(cfg, "cpu")
    layer, out, gr = _run_layer(cfg, p, dy.cuda())
    lg, idx, g = _oracle_route(cfg, h)
    keys = O.selection_keys(lg, h.get("bias"))
    tol = 2 * float(np.abs(np32(layer.buf["logits"]) - lg).max()) + 1e-6
    gidx = layer.buf["topk_idx"].cpu().numpy()
    same = routing_agreement(keys, gidx, idx, tol)
    assert same.all(), "near-tie routing in a small parity case; pick another seed"
    _, saved = O.moe_forward(h["x"], lg, idx, g, h["w1"], h["w3"], h["w2"], _shared(h))
    ref = O.moe_backward(np32(dy), h["x"], lg, idx, g, h["w_gate"], h["w1"], h["w3"], h["w2"], saved, cfg.gate,
                         _shared(h))
    for key in ("dx", "dw1", "dw3", "dw2", "dw_gate", "dg"):
        assert rel(np32(gr[key]), ref[key]) < BF16_TOL, key
    check_rows(np32(gr["dx"]), ref["dx"], BF16_TOL, "dx")
    check_rows(np32(gr["dg"]), ref["dg"], BF16_TOL, "dg")
    dl_ref = np.take_along_axis(ref["dlogits"], idx.astype(np.int64), axis=1)
    assert rel(np32(gr["dlogits"]), dl_ref) < BF16_TOL
    if cfg.n_shared:
        for key in ("dws1", "dws3", "dws2"):
            assert rel(np32(gr[key]), ref[key]) < BF16_TOL, key
    # experts that received no token get exactly zero weight gradients
    counts = O.histogram(idx, cfg.n_exp)
    for ex in np.nonzero(counts == 0)[0]:
        assert not gr["dw1"][ex].any() and not gr["dw3"][ex].any() and not gr["dw2"][ex].any()


def test_update_bias_bitexact():
    for name, mode in (("small_fine", 0), ("small_fine", 1), ("dsv3", 0), ("dsv3", 1)):
        cfg = CONFIGS[name]
        lg = skewed_logits(cfg.n_tok, cfg.n_exp, "zipf").numpy()
        ridx, _ = O.route(lg, None, cfg.top_k, cfg.gate)
        counts = O.histogram(ridx, cfg.n_exp)
        b0 = (np.random.default_rng(3).standard_normal(cfg.n_exp) * 0.01).astype(np.float32)
        bias = torch.from_numpy(b0).cuda()
        d = api.make_desc(cfg)
        for _ in range(3):
            api.moe_update_bias(d, torch.from_numpy(counts).cuda(), bias, 1e-3, mode)
            b0 = O.update_bias(counts, b0, 1e-3, mode)
        np.testing.assert_array_equal(bias.cpu().numpy().view(np.int32), b0.view(np.int32))


# ------------------------------------------------------------- edge cases
EDGE = [
    MoEConfig("one_expert", 130, 128, 128, 1, 1),                                   # E=K=1: dense SwiGLU
    MoEConfig("k_equals_e", 70, 64, 64, 4, 4),                                      # soft MoE
    MoEConfig("single_token", 1, 64, 128, 8, 2),
    MoEConfig("hot_expert", 300, 128, 192, 16, 2, gate="sigmoid", use_bias=True,   # most tokens -> one expert,
              bias_beta=3.0, n_cold=10),                                            # 10 experts empty
]


@pytest.mark.parametrize("cfg", EDGE, ids=lambda c: c.name)
def test_edge_cases(cfg, gemm_form):
    p_cpu = make_layer(cfg, "cpu")
    p, h = to_dev(p_cpu), host_params(p_cpu)
    dy = make_dy(cfg, "cpu")
    layer, out, gr = _run_layer(cfg, p, dy.cuda())
    lg, idx, g = _oracle_route(cfg, h)
    keys = O.selection_keys(lg, h.get("bias"))
    tol = 2 * float(np.abs(np32(layer.buf["logits"]) - lg).max()) + 1e-6
    same = routing_agreement(keys, layer.buf["topk_idx"].cpu().numpy(), idx, tol)
    assert same.all()
    ref, saved = O.moe_forward(h["x"], lg, idx, g, h["w1"], h["w3"], h["w2"], _shared(h))
    check_rows(np32(out), ref, BF16_TOL, "out")
    rg = O.moe_backward(np32(dy), h["x"], lg, idx, g, h["w_gate"], h["w1"], h["w3"], h["w2"], saved, cfg.gate,
                        _shared(h))
    for key in ("dx", "dw1", "dw3", "dw2"):
        assert rel(np32(gr[key]), rg[key]) < BF16_TOL, key
    if np.abs(rg["dw_gate"]).max() > 0:
        assert rel(np32(gr["dw_gate"]), rg["dw_gate"]) < BF16_TOL
    else:
        assert np.abs(np32(gr["dw_gate"])).max() < 1e-6
    counts = O.histogram(idx, cfg.n_exp)
    for ex in np.nonzero(counts == 0)[0]:
        assert not gr["dw1"][ex].any() and not gr["dw2"][ex].any()


def test_graph_capture_replays_identically():
    cfg, p, h = _layer("small_sigmoid")
    dy = make_dy(cfg, "cpu").cuda()
    layer = api.MoELayer(cfg, p, train=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(p["x"], stream=s)        # warm-up outside capture
        layer.backward(dy, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref_out = layer.buf["out"].clone()
    ref_dw1 = layer.grads["dw1"].clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(p["x"])
        layer.backward(dy)
    layer.buf["out"].zero_()
    layer.grads["dw1"].zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.buf["out"], ref_out)
    assert torch.equal(layer.grads["dw1"], ref_dw1)
    assert layer.device_status()[0] == 0
