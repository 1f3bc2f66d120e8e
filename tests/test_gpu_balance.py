"""GPU parity of the load-balancing side path: the auxiliary loss and its
logit gradient, and the load monitor statistics, against the oracle on the
same seeded fp32 logits / routing histograms (routing from the same logits
is bit-exact, so only fp32-vs-fp64 arithmetic separates the two sides)."""
import numpy as np
import pytest
import torch

import oracle as O
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, skewed_logits

pytestmark = pytest.mark.gpu


def _ws(cfg):
    d = api.make_desc(cfg)
    f, _ = api.moe_workspace_size(d)
    ws = torch.empty(f, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    return d, ws


@pytest.mark.parametrize("name,mode", [("tiny", "uniform"), ("small_softmax", "zipf"), ("small_sigmoid", "half0"),
                                       ("small_fine", "uniform"), ("dsv3", "zipf"), ("dsv3", "half0"),
                                       ("mixtral", "uniform")])
def test_aux_loss_and_gradient(name, mode):
    cfg = CONFIGS[name]
    n, e, k = cfg.n_tok, cfg.n_exp, cfg.top_k
    lg = skewed_logits(n, e, mode)
    d, ws = _ws(cfg)
    idx, w = torch.empty(n, k, dtype=torch.int32, device="cuda"), torch.empty(n, k, device="cuda")
    counts, offsets = torch.empty(e, dtype=torch.int32, device="cuda"), torch.empty(e + 1, dtype=torch.int32,
                                                                                     device="cuda")
    bias = torch.zeros(e, device="cuda") if cfg.use_bias else None
    api.moe_route_from_logits(d, lg.cuda(), bias, idx, w, counts, offsets, ws)
    loss = torch.empty(1, device="cuda")
    dl = torch.empty(n, e, device="cuda")
    api.moe_aux_loss(d, lg.cuda(), counts, loss, dl, ws, coef=0.01)
    torch.cuda.synchronize()
    lgh = lg.numpy()
    ridx, _ = O.route(lgh, None if bias is None else np.zeros(e, np.float32), k, cfg.gate)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    want = 0.01 * O.aux_loss(lgh, ridx, e, cfg.gate)
    assert float(loss.item()) == pytest.approx(want, rel=2e-6)
    gw = 0.01 * O.aux_loss_grad(lgh, ridx, e, cfg.gate)
    got = dl.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - gw) / np.linalg.norm(gw) < 1e-5
    assert np.abs(got - gw).max() <= 1e-5 * np.abs(gw).max() + 1e-12


def test_aux_loss_closed_forms_on_gpu():
    """Uniform probabilities and balanced counts give aux = K (E f_i P_i =
    E (K/E)(1/E) per expert); one expert taking every copy with K = 1 and all
    probability mass on it gives E."""
    cfg = CONFIGS["tiny"].replace(n_tok=64, top_k=1)
    d, ws = _ws(cfg)
    e = cfg.n_exp
    loss = torch.empty(1, device="cuda")
    counts = torch.full((e,), 64 // e, dtype=torch.int32, device="cuda")
    api.moe_aux_loss(d, torch.zeros(64, e, device="cuda"), counts, loss, None, ws)
    torch.cuda.synchronize()
    assert float(loss.item()) == pytest.approx(1.0, rel=1e-6)
    lg = torch.full((64, e), -30.0, device="cuda")
    lg[:, 3] = 30.0
    counts = torch.zeros(e, dtype=torch.int32, device="cuda")
    counts[3] = 64
    api.moe_aux_loss(d, lg, counts, loss, None, ws)
    torch.cuda.synchronize()
    assert float(loss.item()) == pytest.approx(e, rel=1e-6)


@pytest.mark.parametrize("e,h", [(8, 1), (8, 100), (256, 37), (1024, 5)])
def test_monitor_stats(e, h):
    g = torch.Generator().manual_seed(40 + e + h)
    hist = torch.randint(0, 50, (h, e), generator=g, dtype=torch.int32)
    hist[:, : e // 8] = 0                                 # some cold experts
    hist[:, -1] += 1                                      # no empty step
    stats = torch.empty(3, device="cuda")
    api.moe_monitor_stats(hist.cuda(), stats)
    torch.cuda.synchronize()
    ref = O.monitor_stats([O.load_stat(row) for row in hist.numpy()], last=h)
    got = stats.cpu().numpy()
    assert got[0] == pytest.approx(ref["min_load"], rel=1e-6, abs=1e-12)
    assert got[1] == pytest.approx(ref["entropy"], rel=1e-6)
    assert int(got[2]) == ref["cold_experts"]
