"""GPU parity of the capacity-factor drop mode (the comparison case of the
dropless layer): the compact maps bit for bit against the oracle from the
same fp32 logits, the layer forward and backward against the oracle's
capacity forward and its backward, and a large factor reproducing the
dropless layer exactly."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import BF16_TOL, host_params, np32, rel, routing_agreement, to_dev
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_dy, make_layer, skewed_logits

pytestmark = pytest.mark.gpu


def _i32(*s):
    return torch.empty(s, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("name,mode,cf", [("tiny", "uniform", 0.5), ("small_softmax", "half0", 1.0),
                                          ("small_fine", "zipf", 1.25), ("dsv3", "zipf", 1.0),
                                          ("dsv3", "half0", 1.25), ("mixtral", "uniform", 1.0)])
def test_capacity_maps_bitexact(name, mode, cf):
    cfg = CONFIGS[name]
    n, e, k, d = cfg.n_tok, cfg.n_exp, cfg.top_k, cfg.d_model
    r = n * k
    desc = api.make_desc(cfg)
    f, _ = api.moe_workspace_size(desc)
    ws = torch.empty(f, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    lg = skewed_logits(n, e, mode)
    idx, w, counts, off = _i32(n, k), torch.empty(n, k, device="cuda"), _i32(e), _i32(e + 1)
    bias = torch.zeros(e, device="cuda") if cfg.use_bias else None
    api.moe_route_from_logits(desc, lg.cuda(), bias, idx, w, counts, off, ws)
    x = torch.randn(n, d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    rf, cf_, ko, roc, cor, xp, nd = _i32(r), _i32(r), _i32(e + 1), _i32(r), _i32(r), \
        torch.empty(r, d, dtype=torch.bfloat16, device="cuda"), _i32(1)
    api.moe_permute_capacity(desc, x.cuda(), idx, off, cf, rf, cf_, ko, roc, cor, xp, nd, ws)
    torch.cuda.synchronize()
    ridx, _ = O.route(lg.numpy(), None if bias is None else np.zeros(e, np.float32), k, cfg.gate)
    cap = O.capacity(n, e, k, cf)
    roc_o, cor_o, kept_o, off_o, nd_o = O.permutation_capacity(ridx, e, cap)
    roc_f, cor_f = O.permutation(ridx, e)
    np.testing.assert_array_equal(rf.cpu().numpy(), roc_f)
    np.testing.assert_array_equal(cf_.cpu().numpy(), cor_f)
    np.testing.assert_array_equal(ko.cpu().numpy(), off_o)
    np.testing.assert_array_equal(roc.cpu().numpy(), roc_o)
    nk = int(off_o[-1])
    np.testing.assert_array_equal(cor.cpu().numpy()[:nk], cor_o)
    assert int(nd.item()) == nd_o
    # kept rows of x_perm are the kept copies' token rows
    xh = x.float().numpy()
    np.testing.assert_array_equal(xp.float().cpu().numpy()[:nk], xh[cor_o // k])
    if mode == "half0" or cf <= 0.5:
        assert nd_o > 0


@pytest.mark.parametrize("name,cf", [("small_softmax", 0.8), ("small_sigmoid", 1.0), ("small_fine", 0.9)])
def test_capacity_layer_forward_backward(name, cf):
    cfg = CONFIGS[name].replace(capacity_factor=cf)
    p_cpu = make_layer(cfg, "cpu")
    p, h = to_dev(p_cpu), host_params(p_cpu)
    dy = make_dy(cfg, "cpu")
    layer = api.MoELayer(cfg, p, train=True)
    out = layer.forward(p["x"])
    gr = layer.backward(dy.cuda())
    torch.cuda.synchronize()
    assert layer.device_status()[0] == 0
    lg = O.gate_logits(h["x"], h["w_gate"])
    idx, g = O.route(lg, h.get("bias"), cfg.top_k, cfg.gate)
    keys = O.selection_keys(lg, h.get("bias"))
    tol = 2 * float(np.abs(np32(layer.buf["logits"]) - lg).max()) + 1e-6
    assert routing_agreement(keys, layer.buf["topk_idx"].cpu().numpy(), idx, tol).all()
    cap = O.capacity(cfg.n_tok, cfg.n_exp, cfg.top_k, cf)
    nd = O.permutation_capacity(idx, cfg.n_exp, cap)[4]
    assert nd > 0 and layer.drop_rate() == pytest.approx(nd / cfg.rows)
    shared = (h["ws1"], h["ws3"], h["ws2"]) if cfg.n_shared else None
    ref, saved = O.moe_forward_capacity(h["x"], lg, idx, g, h["w1"], h["w3"], h["w2"], cap, shared)
    assert rel(np32(out), ref) < BF16_TOL
    rg = O.moe_backward(np32(dy), h["x"], lg, idx, g, h["w_gate"], h["w1"], h["w3"], h["w2"], saved, cfg.gate,
                        shared)
    for key in ("dx", "dw1", "dw3", "dw2", "dw_gate", "dg"):
        assert rel(np32(gr[key]), rg[key]) < BF16_TOL, key
    assert rel(np32(gr["dlogits"]), np.take_along_axis(rg["dlogits"], idx.astype(np.int64), axis=1)) < BF16_TOL


def test_capacity_large_factor_reproduces_dropless_exactly():
    base = CONFIGS["small_sigmoid"]
    p = to_dev(make_layer(base, "cpu"))
    dy = make_dy(base, "cpu").cuda()
    res = []
    for cfg in (base, base.replace(capacity_factor=100.0)):
        layer = api.MoELayer(cfg, p, train=True)
        out = layer.forward(p["x"]).clone()
        gr = {k: v.clone() for k, v in layer.backward(dy).items()}
        torch.cuda.synchronize()
        res.append((out, gr))
        if cfg.capacity_factor:
            assert layer.drop_rate() == 0.0
    assert torch.equal(res[0][0], res[1][0])
    for key in res[0][1]:
        assert torch.equal(res[0][1][key], res[1][1][key]), key
