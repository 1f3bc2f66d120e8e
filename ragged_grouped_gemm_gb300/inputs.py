"""Seeded synthetic inputs for the MoE layer: shapes, seeds, value distributions.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests.  It holds workload definitions and random-number draws only, none of
the layer's arithmetic.

Workloads (from the layer shapes the pages discuss):

* ``tiny``     N=256, D=64, F=128, E=8, K=2, softmax gate, no shared expert.
* ``mixtral``  Mixtral-8x7B-shaped layer: N=4096 (B=2, T=2048), D=4096,
               F=14336, E=8, K=2, softmax gate ([MoE-Eng] §1.1, §4.2).
* ``dsv3``     DeepSeek-V3-shaped fine-grained layer: N=4096, D=7168, F=2048,
               E=256, K=8, sigmoid gate + route bias, one shared expert
               Fs=2048 ([MoE-Eng] §4.3, §5, §6.3, §13.5).  The route bias is
               Zipf-skewed so that loads span 0 to about 8x the mean and some
               experts receive no token.
* ``small_*``  mid-size cases that span several GEMM tiles and ragged tails.

Distributions: x ~ N(0, 1); gate and expert weights ~ N(0, 0.02^2);
upstream gradient dY ~ N(0, 1); all drawn in fp32 from ``torch.Generator``
with fixed seeds and rounded to bf16 (round to nearest even).  No dataset or
trained weight is used: synthetic tokens stand in for activations.
"""
from __future__ import annotations

import dataclasses

import torch

SEEDS = {"x": 1, "w_gate": 2, "w1": 3, "w3": 4, "w2": 5,
         "ws1": 6, "ws3": 7, "ws2": 8, "dy": 9, "bias_perm": 10, "skew": 11}
WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    n_tok: int
    d_model: int
    d_ff: int
    n_exp: int
    top_k: int
    gate: str = "softmax"          # "softmax" | "sigmoid"
    use_bias: bool = False
    n_shared: int = 0
    d_ff_shared: int = 0
    precision: str = "bf16"        # "bf16" | "mxfp8" | "fp8w" (FP8 weights, bf16 activations)
    bias_beta: float = 0.0         # Zipf strength of the route bias
    n_cold: int = 0                # experts whose bias keeps them empty
    capacity_factor: float = 0.0   # > 0: capacity-factor drop mode (comparison case); 0: dropless

    @property
    def rows(self) -> int:
        """Number of token copies N*K (rows of the permuted buffers)."""
        return self.n_tok * self.top_k

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", 256, 64, 128, 8, 2),
    "mixtral": MoEConfig("mixtral", 4096, 4096, 14336, 8, 2),
    # bias_beta: found by bisection with the oracle router on the seeded x and
    # W_g so that the most loaded expert takes 8x the mean load N*K/E (8.0x)
    "dsv3": MoEConfig("dsv3", 4096, 7168, 2048, 256, 8, gate="sigmoid", use_bias=True,
                      n_shared=1, d_ff_shared=2048, bias_beta=0.4833, n_cold=4),
    # profiling case: the Mixtral layer with a quarter of d_ff (about 3 GB on
    # the device, operands still far larger than L2)
    "mixtral_quarter": MoEConfig("mixtral_quarter", 4096, 4096, 3584, 8, 2),
    # profiling case: DeepSeek-V3 expert shapes (~128 rows per expert) on 16
    # experts (0.7 GB of weights, 0.94 GB of fp32 output per weight gradient)
    "dsv3_e16": MoEConfig("dsv3_e16", 256, 7168, 2048, 16, 8, gate="sigmoid", use_bias=True),
    # mid-size parity cases: several tiles in every GEMM dimension, ragged tails
    "small_softmax": MoEConfig("small_softmax", 1000, 256, 384, 8, 2),
    "small_sigmoid": MoEConfig("small_sigmoid", 777, 512, 256, 16, 4, gate="sigmoid",
                               use_bias=True, n_shared=1, d_ff_shared=192,
                               bias_beta=0.6, n_cold=2),
    "small_fine": MoEConfig("small_fine", 513, 384, 128, 64, 8, gate="sigmoid",
                            use_bias=True, n_shared=1, d_ff_shared=256,
                            bias_beta=0.5, n_cold=3),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, std: float = 1.0, device="cpu", chunk_dim0: bool = False):
    """fp32 N(0, std^2) draws from a seeded generator, rounded to bf16.

    With ``chunk_dim0`` the tensor is drawn slice by slice along dim 0 from one
    generator, which bounds the fp32 temporary for very large weights.
    """
    g = _gen(seed, device)
    if not chunk_dim0:
        return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    for i in range(shape[0]):
        out[i] = (torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def route_bias(cfg: MoEConfig, device="cpu") -> torch.Tensor | None:
    """Zipf-skewed route bias: ``b_e = -beta * ln(1 + pi(e))`` with ``pi`` a
    seeded permutation of the experts; the ``n_cold`` lowest-ranked experts get
    -1e4 so that they stay empty.  None when the layer has no bias."""
    if not cfg.use_bias:
        return None
    g = _gen(SEEDS["bias_perm"], "cpu")
    perm = torch.randperm(cfg.n_exp, generator=g)
    ranks = perm.to(torch.float64)
    b = -cfg.bias_beta * torch.log1p(ranks)
    if cfg.n_cold:
        b = torch.where(ranks >= cfg.n_exp - cfg.n_cold, torch.full_like(b, -1e4), b)
    return b.to(torch.float32).to(device)


def make_layer(cfg: MoEConfig, device="cpu") -> dict:
    """All parameters and the input batch of one layer, bf16 on ``device``.

    Keys: x [N,D], w_gate [E,D], w1, w3 [E,F,D], w2 [E,D,F], bias [E] fp32 or
    None, and for a shared expert ws1, ws3 [Fs,D], ws2 [D,Fs].
    """
    big = cfg.n_exp * cfg.d_ff * cfg.d_model > (1 << 26)
    # x and W_g are always drawn on the CPU generator, so the routing of a
    # layer built on any device is the one the oracle computes from the same
    # seeds; the large expert weights are drawn on ``device``.
    t = {
        "x": randn_bf16((cfg.n_tok, cfg.d_model), SEEDS["x"], 1.0, "cpu").to(device),
        "w_gate": randn_bf16((cfg.n_exp, cfg.d_model), SEEDS["w_gate"], WEIGHT_STD, "cpu").to(device),
        "w1": randn_bf16((cfg.n_exp, cfg.d_ff, cfg.d_model), SEEDS["w1"], WEIGHT_STD, device, big),
        "w3": randn_bf16((cfg.n_exp, cfg.d_ff, cfg.d_model), SEEDS["w3"], WEIGHT_STD, device, big),
        "w2": randn_bf16((cfg.n_exp, cfg.d_model, cfg.d_ff), SEEDS["w2"], WEIGHT_STD, device, big),
        "bias": route_bias(cfg, device),
    }
    if cfg.n_shared:
        fs = cfg.d_ff_shared
        t["ws1"] = randn_bf16((fs, cfg.d_model), SEEDS["ws1"], WEIGHT_STD, device)
        t["ws3"] = randn_bf16((fs, cfg.d_model), SEEDS["ws3"], WEIGHT_STD, device)
        t["ws2"] = randn_bf16((cfg.d_model, fs), SEEDS["ws2"], WEIGHT_STD, device)
    return t


def make_dy(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """Upstream gradient dY ~ N(0, 1), bf16 [N, D]."""
    return randn_bf16((cfg.n_tok, cfg.d_model), SEEDS["dy"], 1.0, device)


def skewed_logits(n_tok: int, n_exp: int, mode: str, device="cpu", seed: int = SEEDS["skew"]):
    """fp32 router logits with a prescribed load skew (for routing from logits).

    * ``uniform``  i.i.d. N(0, 1) logits: near-uniform loads.
    * ``zipf``     ``ln p_e + G`` with ``p_e`` proportional to ``1/rank^1`` over a
                   seeded expert ranking and ``G`` standard Gumbel noise; the
                   top-K of these keys draws K distinct experts with Zipf(s=1)
                   preference (heavy experts saturate at one copy per token).
    * ``half0``    i.i.d. N(0, 1) logits, and a seeded half of the tokens gets
                   +20 on expert 0, so expert 0 takes 50% of the tokens.
    * ``ties``     small integers in [-2, 2]: many exact ties.
    """
    g = _gen(seed, "cpu")
    if mode == "uniform":
        lg = torch.randn((n_tok, n_exp), generator=g, dtype=torch.float32)
    elif mode == "zipf":
        perm = torch.randperm(n_exp, generator=g).to(torch.float64)
        logp = -torch.log1p(perm)                      # ln(1/rank), rank = perm + 1
        u = torch.rand((n_tok, n_exp), generator=g, dtype=torch.float64).clamp_(1e-12, 1 - 1e-12)
        lg = (logp[None, :] - torch.log(-torch.log(u))).to(torch.float32)
    elif mode == "half0":
        lg = torch.randn((n_tok, n_exp), generator=g, dtype=torch.float32)
        pick = torch.randperm(n_tok, generator=g)[: n_tok // 2]
        lg[pick, 0] += 20.0
    elif mode == "ties":
        lg = torch.randint(-2, 3, (n_tok, n_exp), generator=g).to(torch.float32)
    else:
        raise ValueError(mode)
    return lg.to(device)


def sample_tokens(n_tok: int, n: int, seed: int = 12) -> torch.Tensor:
    """A seeded sorted sample of ``n`` distinct token indices (all if n >= n_tok)."""
    if n >= n_tok:
        return torch.arange(n_tok)
    g = _gen(seed, "cpu")
    return torch.randperm(n_tok, generator=g)[:n].sort().values
