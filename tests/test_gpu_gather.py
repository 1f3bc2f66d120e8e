"""The dispatch fused into GEMM1's operand loads ("LLM Infrastructure
Engineering 08: MoE Training Engineering" §9 engineering notes: scatter +
grouped GEMM): moe_grouped_ffn_gather reads each expert's rows straight from
the token matrix through copy_of_row (TMA four-row gathers) instead of a
permuted copy.  The tile contents the tensor cores see are the same rows in
the same order, so its outputs must equal moe_grouped_ffn's bit for bit; the
inference layer built on it is also checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import BF16_TOL, check_rows, host_params, np32, routing_agreement, to_dev
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_layer

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "small_softmax", "small_sigmoid", "small_fine"]


@pytest.fixture(params=["1", "0"], ids=["cta_pair", "one_sm"])
def gemm_form(request, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", request.param)
    return request.param


def _both_ffns(cfg, p):
    """Route with the layer's own gate, then run the grouped FFN once from
    x_perm (moe_permute + moe_grouped_ffn) and once gathered
    (moe_permute_maps + moe_grouped_ffn_gather); return both outputs."""
    n, d, f, e, k = cfg.n_tok, cfg.d_model, cfg.d_ff, cfg.n_exp, cfg.top_k
    r, fs, sh = cfg.rows, cfg.d_ff_shared, cfg.n_shared
    desc = api.make_desc(cfg)
    _, wsb = api.moe_workspace_size(desc)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    z = lambda *s, dt=torch.bfloat16: torch.zeros(s, dtype=dt, device="cuda")   # noqa: E731
    lg, idx, w, cnt, off = z(n, e, dt=torch.float32), z(n, k, dt=torch.int32), z(n, k, dt=torch.float32), \
        z(e, dt=torch.int32), z(e + 1, dt=torch.int32)
    api.moe_route(desc, p["x"], p["w_gate"], p.get("bias"), lg, idx, w, cnt, off, ws)
    outs = []
    for mode in ("x_perm", "gather"):
        roc, cor = z(r, dt=torch.int32), z(r, dt=torch.int32)
        a1, a3, h, y = z(r, f), z(r, f), z(r, f), z(r, d)
        a1s, a3s, hs, ys = (z(n, fs), z(n, fs), z(n, fs), z(n, d)) if sh else (None,) * 4
        if mode == "x_perm":
            xp = z(r, d)
            api.moe_permute(desc, p["x"], idx, off, roc, cor, xp, ws)
            api.moe_grouped_ffn(desc, xp, off, p["x"], p["w1"], p["w3"], p["w2"], p.get("ws1"), p.get("ws3"),
                                p.get("ws2"), a1, a3, h, a1s, a3s, hs, y, ys, ws)
        else:
            api.moe_permute_maps(desc, idx, off, roc, cor, ws)
            api.moe_grouped_ffn_gather(desc, p["x"], cor, off, p["w1"], p["w3"], p["w2"], p.get("ws1"),
                                       p.get("ws3"), p.get("ws2"), a1, a3, h, a1s, a3s, hs, y, ys, ws)
        torch.cuda.synchronize()
        bits, site = api.moe_get_device_status(ws)
        assert bits == 0, f"device status {bits} (site {site})"
        outs.append({"row_of_copy": roc, "copy_of_row": cor, "a1": a1, "a3": a3, "h": h, "y_perm": y,
                     "hs": hs, "y_shared": ys})
    return outs


def _assert_same(a, b):
    for key in a:
        if a[key] is None:
            continue
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key]), key


@pytest.mark.parametrize("name", SMALL)
def test_gathered_ffn_equals_permuted_ffn_bitwise(name, gemm_form):
    cfg = CONFIGS[name]
    p = to_dev(make_layer(cfg, "cpu"))
    ref, got = _both_ffns(cfg, p)
    _assert_same(ref, got)


@pytest.mark.parametrize("name", SMALL)
def test_inference_layer_with_gathered_ffn_matches_oracle(name):
    cfg = CONFIGS[name]
    p_cpu = make_layer(cfg, "cpu")
    p, h = to_dev(p_cpu), host_params(p_cpu)
    layer = api.MoELayer(cfg, p, train=False, gather=True)
    assert layer.gather and layer.buf["x_perm"] is None
    out = layer.forward(p["x"])
    torch.cuda.synchronize()
    assert layer.device_status()[0] == 0
    lg = O.gate_logits(h["x"], h["w_gate"])
    idx, g = O.route(lg, h.get("bias"), cfg.top_k, cfg.gate)
    keys = O.selection_keys(lg, h.get("bias"))
    tol = 2 * float(np.abs(np32(layer.buf["logits"]) - lg).max()) + 1e-6
    same = routing_agreement(keys, layer.buf["topk_idx"].cpu().numpy(), idx, tol)
    shared = (h["ws1"], h["ws3"], h["ws2"]) if cfg.n_shared else None
    ref, _ = O.moe_forward(h["x"], lg, idx, g, h["w1"], h["w3"], h["w2"], shared)
    check_rows(np32(out)[same], ref[same], BF16_TOL, "out")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_gathered_forward_full_size_equals_permuted_forward(name):
    """Full-size inference forward (the launch configuration of the bench's
    inference timing): the gathered layer's output equals the output of the
    layer that materialises x_perm, bit for bit."""
    cfg = CONFIGS[name]
    torch.cuda.empty_cache()
    p = make_layer(cfg, "cuda")
    ref = api.MoELayer(cfg, p, train=False)
    assert not ref.gather and ref.buf["x_perm"] is not None
    out_ref = ref.forward(p["x"]).clone()
    del ref
    layer = api.MoELayer(cfg, p, train=False, gather=True)
    assert layer.gather
    out = layer.forward(p["x"])
    torch.cuda.synchronize()
    assert layer.device_status()[0] == 0
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
    del layer, p
    torch.cuda.empty_cache()
