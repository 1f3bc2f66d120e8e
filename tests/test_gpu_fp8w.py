"""GPU parity of the FP8-weight mode (E4M3 weights with one fp32 scale per
128 x 128 tile, bf16 activations): the tile quantiser bit for bit against
the oracle, and the layer forward and backward against the bf16 oracle run
on the dequantised weights (normwise 5e-3: the only differences left are
those of the bf16 path)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import BF16_TOL, host_params, np32, rel, routing_agreement, to_dev
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_dy, make_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(3, 200, 304), (1, 128, 128), (2, 64, 1040)])
def test_fp8_tile_quantise_bitexact(shape):
    g = torch.Generator().manual_seed(60 + shape[1])
    w = torch.randn(shape, generator=g) * torch.logspace(-6, 6, shape[2])[None, None, :]
    w[0, :64, :64] = 0.0                                   # an all-zero corner
    wb = w.to(torch.bfloat16)
    q = api.quantize_weights_fp8_tile({"w1": wb.cuda()})
    torch.cuda.synchronize()
    rc, rs = O.fp8_tile_quantize(wb.float().numpy())
    np.testing.assert_array_equal(q["w1"].cpu().numpy(), rc)
    np.testing.assert_array_equal(q["w1_scale"].cpu().numpy().view(np.uint32), rs.view(np.uint32))


def _deq(h, key):
    c, s = O.fp8_tile_quantize(h[key])
    return O.fp8_tile_dequantize(c, s)


@pytest.mark.parametrize("name", ["tiny", "small_softmax", "small_sigmoid", "small_fine"])
def test_fp8w_layer_forward_backward(name):
    cfg = CONFIGS[name].replace(precision="fp8w")
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
    w1, w3, w2 = _deq(h, "w1"), _deq(h, "w3"), _deq(h, "w2")
    shared = (_deq(h, "ws1"), _deq(h, "ws3"), _deq(h, "ws2")) if cfg.n_shared else None
    ref, saved = O.moe_forward(h["x"], lg, idx, g, w1, w3, w2, shared)
    assert rel(np32(out), ref) < BF16_TOL
    plain, _ = O.moe_forward(h["x"], lg, idx, g, h["w1"], h["w3"], h["w2"],
                             (h["ws1"], h["ws3"], h["ws2"]) if cfg.n_shared else None)
    assert rel(np32(out), plain) > 2e-3                     # the FP8 weights are visible
    rg = O.moe_backward(np32(dy), h["x"], lg, idx, g, h["w_gate"], w1, w3, w2, saved, cfg.gate, shared)
    for key in ("dx", "dw1", "dw3", "dw2", "dw_gate", "dg"):
        assert rel(np32(gr[key]), rg[key]) < BF16_TOL, key
    if cfg.n_shared:
        for key in ("dws1", "dws3", "dws2"):
            assert rel(np32(gr[key]), rg[key]) < BF16_TOL, key
