"""The kernel-timing entry points on the GPU: every grouped-GEMM launch of a
forward + backward is timed under its kind, launches past the event pool
and launches under graph capture are counted as untimed, and timing does
not change results.  With E <= 32 experts the router runs as one fused
kernel (no logits GEMM, so nothing under "gate"); above that the logits
GEMM is one "gate" launch."""
import pytest
import torch

from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_dy, make_layer

pytestmark = pytest.mark.gpu


def _layer(name):
    cfg = CONFIGS[name]
    p = make_layer(cfg, "cpu")
    p = {k: (v.cuda() if v is not None else None) for k, v in p.items()}
    return cfg, p, api.MoELayer(cfg, p, train=True), make_dy(cfg, "cpu").cuda()


@pytest.mark.parametrize("name", ["small_sigmoid", "small_softmax", "small_fine"])
def test_every_grouped_gemm_is_timed_under_its_kind(name):
    cfg, p, layer, dy = _layer(name)
    layer.forward(p["x"])
    layer.backward(dy)
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in layer.grads.items()}
    api.moe_timing_enable(64)
    try:
        layer.forward(p["x"])
        layer.backward(dy)
        torch.cuda.synchronize()
        sets = 2 if cfg.n_shared else 1               # routed experts (+ the shared expert)
        want = {"ffn_fwd": 2 * sets, "dgrad": 2 * sets, "wgrad": 3 * sets}
        for kind, n in want.items():
            ms, timed, untimed = api.moe_timing_read(kind)
            assert (timed, untimed) == (n, 0), kind
            assert 0.0 < ms < 1e3, kind
        ms, timed, untimed = api.moe_timing_read("gate")   # the router logits GEMM (E > 32)
        if cfg.n_exp > 32:
            assert (timed, untimed) == (1, 0) and 0.0 < ms < 1e3
        else:
            assert (timed, untimed) == (0, 0)
    finally:
        api.moe_timing_disable()
    for k, v in layer.grads.items():
        assert torch.equal(v, ref[k]), k
    assert layer.device_status()[0] == 0


def test_pool_overflow_and_graph_capture_are_untimed():
    cfg, p, layer, dy = _layer("small_fine")   # E = 64: the router's logits GEMM is a grouped-GEMM launch
    assert cfg.n_exp > 32 and cfg.n_shared
    layer.forward(p["x"])
    torch.cuda.synchronize()
    api.moe_timing_enable(2)
    try:
        layer.forward(p["x"])                          # router launches + 4 expert GEMMs; only 2 slots
        torch.cuda.synchronize()
        g_ms, g_n, g_u = api.moe_timing_read("gate")
        f_ms, f_n, f_u = api.moe_timing_read("ffn_fwd")
        assert (g_n, g_u, f_n, f_u) == (1, 0, 1, 3)
        api.moe_timing_enable(64)                       # clears the records
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.forward(p["x"])
        graph.replay()
        torch.cuda.synchronize()
        assert api.moe_timing_read("ffn_fwd")[1:] == (0, 4)
        assert api.moe_timing_read("gate")[1:] == (0, 1)
    finally:
        api.moe_timing_disable()
    assert layer.device_status()[0] == 0
