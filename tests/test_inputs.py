"""The seeded workloads have the structure their descriptions state.

DeepSeek-V3-shaped layer: the Zipf-skewed route bias makes the loads span 0
to about 8x the mean N*K/E, with some experts empty (the load skew of the
fine-grained layer, "LLM Infrastructure Engineering 08: MoE Training
Engineering" §6.3 bias-adjusted selection on a §13.5 fine-grained layer).
The loads are those of the oracle router on the seeded x and W_g, which
every device draws from the same CPU generator."""
import numpy as np

import oracle as O
from ragged_grouped_gemm_gb300.inputs import CONFIGS, SEEDS, WEIGHT_STD, make_layer, randn_bf16, route_bias


def test_dsv3_route_bias_spans_zero_to_8x_mean():
    cfg = CONFIGS["dsv3"]
    x = randn_bf16((cfg.n_tok, cfg.d_model), SEEDS["x"], 1.0, "cpu").float().numpy()
    wg = randn_bf16((cfg.n_exp, cfg.d_model), SEEDS["w_gate"], WEIGHT_STD, "cpu").float().numpy()
    idx, _ = O.route(O.gate_logits(x, wg), route_bias(cfg).numpy(), cfg.top_k, cfg.gate)
    counts = O.histogram(idx, cfg.n_exp)
    ratio = counts.max() / (cfg.rows / cfg.n_exp)
    assert abs(ratio - 8.0) <= 0.05 * 8.0, ratio
    assert (counts == 0).sum() >= cfg.n_cold


def test_x_and_gate_weights_do_not_depend_on_the_device_generator():
    """make_layer draws x and W_g from the CPU generator whatever the device,
    so a layer built on the GPU routes like the oracle on the same seeds."""
    import torch
    cfg = CONFIGS["tiny"]
    a = make_layer(cfg, "cpu")
    b = make_layer(cfg, torch.device("cpu"))
    assert torch.equal(a["x"], b["x"]) and torch.equal(a["w_gate"], b["w_gate"])
