"""Benchmark of the dropless MoE layer (forward + backward) on GB300.

One step = one pass of the whole hot path over one batch: router (gate GEMM,
top-K, histogram, scan), permute, grouped SwiGLU FFN, combine, then the
backward (combine backward, grouped data and weight gradients, router
gradient, input gradient).  Default workload: the Mixtral-8x7B-shaped layer
(N=4096 tokens, D=4096, F=14336, E=8, K=2, softmax gate), synthetic seeded
inputs.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs an
independent replica on its own tokens (the layer has no exchange step on one
GPU per replica), timing is max over ranks and `value` counts all ranks'
tokens.  `--impl reference` times the CPU oracle on the machine's host cores on a
bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s fwd+bwd (grouped-GEMM TFLOP/s, % peak reported alongside), 1 GB300"
PROFILES = os.path.join(ROOT, "profiles")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--sample", type=int, default=0, help="oracle token sample (0: automatic)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-configs", action="store_true",
                    help="time only the chosen workload (by default the Mixtral bf16 run is followed by the "
                         "DeepSeek-V3 bf16 and MXFP8 and the Mixtral MXFP8 layers, reported as sub_results)")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "mxfp8", "fp8w"],
                    help="expert GEMM operands: bf16; MXFP8 (E4M3 codes, E8M0 scales per 32 along the contraction,"
                         " forward and backward); fp8w (E4M3 weights with fp32 scales per 128x128 tile)")
    ap.add_argument("--sweep", action="store_true",
                    help="load-skew sweep: forward and forward+backward for bf16, MXFP8, FP8 weights and the "
                         "capacity-factor mode (prints one JSON line of results)")
    return ap.parse_args()


def flops(cfg) -> dict:
    """Algorithmic FLOPs of one step: 6DF per routed copy forward and 12DF
    backward (no padding, empty experts cost nothing), the same per token for
    the shared expert, 2DE / 4DE per token for the router."""
    n, k, d, f, e = cfg.n_tok, cfg.top_k, cfg.d_model, cfg.d_ff, cfg.n_exp
    fs = cfg.d_ff_shared * cfg.n_shared
    return {"ffn_fwd": 6 * n * k * d * f + 6 * n * d * fs, "router_fwd": 2 * n * d * e,
            "ffn_bwd": 12 * n * k * d * f + 12 * n * d * fs, "router_bwd": 4 * n * d * e}


def ffn_bytes(cfg, nonempty: int) -> int:
    """Algorithmic HBM bytes of one grouped-FFN call (training forward):
    GEMM1 reads x_perm and w1, w3 of the experts that received tokens and
    writes h, a1, a3; GEMM2 reads h and w2 and writes y_perm; the shared expert
    does the same over all tokens.  MXFP8: operands are E4M3 codes plus one
    E8M0 scale per 32 (1 + 1/32 bytes per element), GEMM1 also writes the
    quantised h that GEMM2 reads; fp8w: weights are E4M3 plus one fp32 scale
    per 128 x 128 tile."""
    n, k, d, f = cfg.n_tok, cfg.top_k, cfg.d_model, cfg.d_ff
    r = n * k
    q = 1 + 1 / 32
    wb = {"bf16": 2, "mxfp8": q, "fp8w": 1 + 4 / 128 ** 2}[cfg.precision]

    def pair(rows, experts, ff):
        if cfg.precision == "mxfp8":
            g1 = q * rows * d + wb * 2 * experts * ff * d + 2 * 3 * rows * ff + q * rows * ff
            g2 = q * rows * ff + wb * experts * d * ff + 2 * rows * d
        else:
            g1 = 2 * rows * d + wb * 2 * experts * ff * d + 2 * 3 * rows * ff
            g2 = 2 * rows * ff + wb * experts * d * ff + 2 * rows * d
        return g1 + g2
    b = pair(r, nonempty, f)
    if cfg.n_shared:
        b += pair(n, 1, cfg.d_ff_shared)
    return int(b)


def workload_name(cfg) -> str:
    """The workload string of the `config` key (both arms)."""
    return (f"{cfg.name}: N={cfg.n_tok} D={cfg.d_model} F={cfg.d_ff} E={cfg.n_exp} K={cfg.top_k} {cfg.gate}"
            + (" +route bias" if cfg.use_bias else "") + (f" +shared Fs={cfg.d_ff_shared}" if cfg.n_shared else "")
            + ", fwd+bwd" + ("" if cfg.precision == "bf16" else f", {cfg.precision} expert GEMMs"))


def kind_work(cfg, kind: str, nonempty: int) -> tuple[float, float]:
    """Algorithmic FLOPs and HBM bytes of one step's grouped GEMMs of one
    timing kind.  Operand bytes are 2 (bf16), 1 + 1/32 (MXFP8 codes and
    scales) or, for fp8w weights, 1 + 4/128^2; the weight gradients are
    written in fp32 for every expert (zeros for the empty ones)."""
    n, k, d, f, e = cfg.n_tok, cfg.top_k, cfg.d_model, cfg.d_ff, cfg.n_exp
    r, fs = n * k, cfg.d_ff_shared if cfg.n_shared else 0
    act = 1 + 1 / 32 if cfg.precision == "mxfp8" else 2
    wt = {"bf16": 2, "mxfp8": 1 + 1 / 32, "fp8w": 1 + 4 / 128 ** 2}[cfg.precision]
    fl = flops(cfg)
    if kind == "gate":
        return fl["router_fwd"], 2 * n * d + 2 * e * d + 4 * n * e
    if kind == "ffn_fwd":
        return fl["ffn_fwd"], ffn_bytes(cfg, nonempty)
    sets = [(r, nonempty, e, f)] + ([(n, 1, 1, fs)] if fs else [])
    if kind == "dgrad":
        # through w2 (+ SwiGLU derivative: reads dYw, w2, a1, a3; writes da1, da3), then through w1|w3
        # (reads da1, da3, w1, w3; writes dx_perm)
        b = sum(act * rows * d + wt * ne * d * ff + 2 * 4 * rows * ff + act * 2 * rows * ff + wt * 2 * ne * ff * d
                + 2 * rows * d for rows, ne, _, ff in sets)
        return fl["ffn_bwd"] / 2, b
    # wgrad: dW2 = dYw^T h, dW1 = da1^T x, dW3 = da3^T x, each reading both operands once
    b = sum(3 * 4 * ee * d * ff + 3 * act * rows * (d + ff) for rows, _, ee, ff in sets)
    return fl["ffn_bwd"] / 2, b


def aggregate(world: int, tokens_per_step: int, steps: int, ms_local: float, reduce_max) -> tuple[float, float]:
    """Whole-job throughput of `world` replicas: every rank processes
    `tokens_per_step` tokens per step; the job takes the slowest rank's time.
    Returns (tokens/s over all ranks, max milliseconds)."""
    ms = reduce_max(ms_local) if world > 1 else ms_local
    return world * tokens_per_step * steps / (ms / 1e3), ms


def route_launches(cfg) -> int:
    """moe_route's kernels: one fused router kernel for E <= 32; otherwise
    dense offsets, the router logits GEMM, and one kernel for the ordered sum
    of the GEMM's contraction slices, top-K, histogram and scan."""
    return 1 if cfg.n_exp <= 32 else 3


def fused_dispatch(cfg) -> bool:
    """Whether the layer routes and permutes in one call (moe_route_permute)."""
    return cfg.n_exp <= 32 and cfg.precision != "mxfp8" and cfg.capacity_factor <= 0


def launches_per_step(cfg) -> int:
    """Kernels libmoe launches for one forward + backward (see moe_api.cu)."""
    from ragged_grouped_gemm_gb300 import _lib  # noqa: F401  (ensures the library is the one counted)
    # permute: one launch while ceil(N/16) * E <= 131072; else the token-chunked map kernels + rows
    sp = -(-cfg.n_tok // 16) * cfg.n_exp <= 131072
    maps = 1 if cfg.rows <= 65536 else 3   # map kernels: one CTA up to 65536 copies, else token-chunked
    if cfg.precision == "mxfp8":
        # route; permute (quantising; one launch, else maps + row quantiser + token quantiser for the shared
        # expert); grouped FFN: GEMM1, GEMM2 (+ token quantiser if the permute did not quantise them,
        # dense offsets, GEMM1, GEMM2); combine
        fwd = route_launches(cfg) + (1 if sp else maps + 1 + (1 if cfg.n_shared else 0)) + 2 + 1
        fwd += 3 if cfg.n_shared else 0
        # per expert set: row-wise quantisers of dYw (fused into the combine backward for the routed
        # experts), da1, da3; pad offsets, 5 transposing quantisers, 5 GEMMs
        per_set = 2 + 1 + 5 + 5
        bwd = 1 + per_set + (1 + per_set + 1 if cfg.n_shared else 0) + 3 + 1   # + combine bwd, router grad, unpermute
        return fwd + bwd + (1 if cfg.use_bias else 0)
    # route and permute (one fused launch for E <= 32; else route, then one permute launch or maps + rows);
    # GEMM1, GEMM2; combine
    disp = 1 if fused_dispatch(cfg) else route_launches(cfg) + (1 if sp else maps + 1)
    fwd = disp + 2 + 1
    if cfg.n_shared:
        fwd += 3
    # combine bwd; dgrad2, wgrad2, dgrad1, wgrad1, wgrad3 (each weight gradient over several
    # experts preceded by the kernel that writes their per-group tensor maps); unpermute-sum
    bwd = 1 + 5 + (3 if cfg.n_exp > 1 else 0) + 1
    if cfg.n_shared:
        bwd += 6
    bwd += 3                     # router weight gradient: chunk prefix, chunk partials, reduction
    return fwd + bwd + (1 if cfg.use_bias else 0)      # route-bias update


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [line for line in out.splitlines() if line.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        loaded = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a stored ncu capture, or None when absent or
    when the kernel source has changed since the capture."""
    path = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(f"{kernel}@{workload}")
    if not rec:
        return None
    src = os.path.join(ROOT, "ragged_grouped_gemm_gb300", "csrc", rec["source"])
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["source_sha"]:
        return None
    return rec["bytes_per_launch"]


# ----------------------------------------------------------------- oracle arm
def oracle_step_sample(cfg, host, sample_idx, dy_host):
    """Forward + backward of the CPU oracle on a token sample (its own routing);
    the MXFP8 oracle for MXFP8 operands (fp8w: `host` holds the dequantised
    weights, prepared once outside the timed step as on the GPU side)."""
    import oracle as O
    x = host["x"][sample_idx]
    dy = dy_host[sample_idx]
    shared = (host["ws1"], host["ws3"], host["ws2"]) if cfg.n_shared else None
    lg = O.gate_logits(x, host["w_gate"])
    idx, g = O.route(lg, host.get("bias"), cfg.top_k, cfg.gate)
    if cfg.precision == "mxfp8":
        out, saved = O.moe_forward_mxfp8(x, idx, g, host["w1"], host["w3"], host["w2"], shared, return_saved=True)
        O.moe_backward_mxfp8(dy, x, lg, idx, g, host["w_gate"], host["w1"], host["w3"], host["w2"], saved, cfg.gate,
                             shared)
        return out
    out, saved = O.moe_forward(x, lg, idx, g, host["w1"], host["w3"], host["w2"], shared)
    O.moe_backward(dy, x, lg, idx, g, host["w_gate"], host["w1"], host["w3"], host["w2"], saved, cfg.gate, shared)
    return out


def time_oracle(cfg, sample: int, steps: int = 1):
    import numpy as np
    import torch

    from ragged_grouped_gemm_gb300.inputs import make_dy, make_layer, sample_tokens
    p = make_layer(cfg, "cpu")
    host = {k: (v.float().numpy() if v is not None else None) for k, v in p.items()}
    dy = make_dy(cfg, "cpu").float().numpy()
    del p
    if cfg.precision == "fp8w":
        import oracle as O
        for key in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
            if host.get(key) is not None:
                host[key] = O.fp8_tile_dequantize(*O.fp8_tile_quantize(host[key]))
    idx = sample_tokens(cfg.n_tok, sample).numpy()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle_step_sample(cfg, host, idx, dy)
        times.append(time.perf_counter() - t0)
    del torch, np
    return len(idx), times


# ----------------------------------------------------------------- GPU arm
def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from ragged_grouped_gemm_gb300 import api
    from ragged_grouped_gemm_gb300.inputs import make_dy, make_layer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    p = make_layer(cfg, dev)
    dy = make_dy(cfg, dev)
    layer = api.MoELayer(cfg, p, train=True, device=dev)
    b, d, ws = layer.buf, layer.desc, layer.ws
    x = p["x"]
    # E <= 32 with bf16 rows: routing and dispatch are one call (moe_route_permute), as the layer runs them
    fused = layer.fused_dispatch
    names = (["route_permute"] if fused else ["route", "permute"]) + ["grouped_ffn", "combine", "backward"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[names.index(i) if isinstance(i, str) else i].record()
        mark(0)
        if fused:
            api.moe_route_permute(d, x, p["w_gate"], p.get("bias"), b["logits"], b["topk_idx"], b["topk_w"],
                                  b["counts"], b["offsets"], b["row_of_copy"], b["copy_of_row"], b["x_perm"], ws)
        else:
            api.moe_route(d, x, p["w_gate"], p.get("bias"), b["logits"], b["topk_idx"], b["topk_w"], b["counts"],
                          b["offsets"], ws)
            mark(1)
            if layer.mx:
                api.moe_permute_mxfp8(d, x, b["topk_idx"], b["offsets"], b["row_of_copy"], b["copy_of_row"],
                                      b["xq_perm"], b["xs_perm"], b["xq_tok"], b["xs_tok"], ws)
            else:
                api.moe_permute(d, x, b["topk_idx"], b["offsets"], b["row_of_copy"], b["copy_of_row"],
                                b["x_perm"], ws)
        mark("grouped_ffn")
        saved = {key: b[key] for key in ("a1", "a3", "h", "a1s", "a3s", "hs") if b.get(key) is not None}
        if layer.mx:
            api.moe_grouped_ffn_mxfp8(d, b["xq_perm"], b["xs_perm"], b["offsets"], b["xq_tok"], b["xs_tok"],
                                      layer.wq, saved, b["y_perm"], b["y_shared"], ws)
        elif layer.w8:
            api.moe_grouped_ffn_fp8w(d, b["x_perm"], b["offsets"], x, layer.w8q, saved, b["y_perm"], b["y_shared"],
                                     ws)
        else:
            api.moe_grouped_ffn(d, b["x_perm"], b["offsets"], x, p["w1"], p["w3"], p["w2"], p.get("ws1"),
                                p.get("ws3"), p.get("ws2"), b["a1"], b["a3"], b["h"], b["a1s"], b["a3s"], b["hs"],
                                b["y_perm"], b["y_shared"], ws)
        mark("combine")
        api.moe_combine(d, b["y_perm"], b["row_of_copy"], b["topk_w"], b["y_shared"], b["out"])
        mark("backward")
        layer.x = x
        layer.backward(dy)
        mark(len(names))
        if cfg.use_bias:
            layer.update_bias(1e-3, 0)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bits, site = layer.device_status()
    if bits:
        raise RuntimeError(f"device status {bits} at site {site}")

    # --- device-timed fwd+bwd steps (inputs resident in HBM)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local_rank).__enter__()   # sampled over all three timed loops
    api.moe_timing_enable(64 * args.steps + 64)   # CUDA events around every grouped GEMM of the timed steps
    t0.record()
    for i in range(args.steps):
        step(evs[i])
    t1.record()
    torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1)
    # per call: the median over the timed steps.  The first timed step starts
    # on an idle GPU, so its first calls also hold the host's time to issue
    # them; in the later steps the host is ahead and the events see GPU time.
    per_call = {n: statistics.median(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                for j, n in enumerate(names)}
    kernels = {}
    for kind in api.TIMING_KINDS:
        k_ms, k_n, k_u = api.moe_timing_read(kind)
        if k_u:
            raise RuntimeError(f"{k_u} untimed {kind} launches")
        kernels[kind] = {"ms_total": k_ms, "launches": k_n}
    api.moe_timing_disable()

    # --- forward-only steps
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record()
    for _ in range(args.steps):
        layer.forward(x)
    f1.record()
    torch.cuda.synchronize()
    ms_fwd = f0.elapsed_time(f1)

    # --- end to end through the public API with pinned host buffers.  Every
    # step uploads its inputs (x, dY) from pinned host memory and downloads
    # its results (output, input gradient) to it, all inside the timed region.
    # The copies run on a copy stream as a training loop's prefetch would:
    # step i+1's uploads and step i's downloads overlap step i+1's compute.
    # Inputs and results are double-buffered; the results are first staged
    # on the device (two 16-byte-row copies) so the next step may overwrite
    # the layer's own output buffers.
    hx = x.cpu().pin_memory()
    hdy = dy.cpu().pin_memory()
    hout = [torch.empty(b["out"].shape, dtype=b["out"].dtype).pin_memory() for _ in range(2)]
    hdx = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for _ in range(2)]
    x_in = [torch.empty_like(x) for _ in range(2)]
    dy_in = [torch.empty_like(dy) for _ in range(2)]
    out_st = [torch.empty_like(b["out"]) for _ in range(2)]
    dx_st = [torch.empty_like(x) for _ in range(2)]
    comp = torch.cuda.current_stream()
    cs = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up, used, staged, down = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(comp)
    cs.wait_event(e0)

    def upload(j):
        with torch.cuda.stream(cs):
            x_in[j].copy_(hx, non_blocking=True)
            dy_in[j].copy_(hdy, non_blocking=True)
            up[j].record(cs)

    upload(0)
    for i in range(args.steps):
        j = i % 2
        if i + 1 < args.steps:
            if i >= 1:
                cs.wait_event(used[1 - j])       # step i-1 is done with the other input buffers
            upload(1 - j)
        comp.wait_event(up[j])
        layer.forward(x_in[j])
        grads = layer.backward(dy_in[j])
        if cfg.use_bias:
            layer.update_bias(1e-3, 0)
        used[j].record(comp)
        if i >= 2:
            comp.wait_event(down[j])             # step i-2's download has left this staging buffer
        out_st[j].copy_(b["out"], non_blocking=True)
        dx_st[j].copy_(grads["dx"], non_blocking=True)
        staged[j].record(comp)
        with torch.cuda.stream(cs):
            cs.wait_event(staged[j])
            hout[j].copy_(out_st[j], non_blocking=True)   # the step's results: output and input gradient
            hdx[j].copy_(dx_st[j], non_blocking=True)
            down[j].record(cs)
    comp.wait_stream(cs)
    e1.record(comp)
    torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    bits, site = layer.device_status()
    if bits:
        raise RuntimeError(f"device status {bits} at site {site}")

    # --- MXFP8: the expert weights' E4M3 codes (rowwise for the forward,
    # columnwise for the data gradients) are made once per weight update,
    # outside the layer's forward + backward, so they are not in the step;
    # their cost is timed here on its own (median of three updates)
    weight_quant_ms = None
    if cfg.precision == "mxfp8":
        wq_ms = []
        for _ in range(3):
            q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            q0.record()
            wq = api.quantize_weights_mxfp8(p)
            wqt = api.quantize_weights_mxfp8_t(p)
            q1.record()
            torch.cuda.synchronize()
            wq_ms.append(q0.elapsed_time(q1))
            del wq, wqt
        weight_quant_ms = sorted(wq_ms)[1]
        torch.cuda.empty_cache()

    # --- inference forward (no saved activations), GEMM1 rows gathered from x
    # (moe_permute_maps + moe_grouped_ffn_gather) against the same layer with a
    # permuted copy of the tokens (moe_permute + moe_grouped_ffn)
    inference = None
    if cfg.precision == "bf16" and cfg.capacity_factor <= 0:
        del layer
        torch.cuda.empty_cache()
        inference = {}
        for mode in ("gather", "x_perm"):
            inf = api.MoELayer(cfg, p, train=False, device=dev, gather=mode == "gather")
            for _ in range(args.warmup):
                inf.forward(x)
            i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            i0.record()
            for _ in range(args.steps):
                inf.forward(x)
            i1.record()
            torch.cuda.synchronize()
            inference[mode] = cfg.n_tok * args.steps / (i0.elapsed_time(i1) / 1e3)
            assert inf.device_status()[0] == 0
            del inf
            torch.cuda.empty_cache()
        layer = None

    def max_over_ranks(v):
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    nonempty = int((b["counts"] > 0).sum().item())
    counts = b["counts"].float()
    res = {"cfg": cfg, "per_call": per_call, "kernels": kernels, "clocks": clk.summary(), "nonempty": nonempty,
           "inference_fwd": inference, "weight_quant_ms": weight_quant_ms,
           "max_load_over_mean": float(counts.max()) / (cfg.rows / cfg.n_exp),
           "h2d": hx.numel() * 2 + hdy.numel() * 2, "d2h": hout[0].numel() * 2 + hdx[0].numel() * 2}
    for key, v in (("step", ms), ("fwd", ms_fwd), ("e2e", ms_e2e)):
        res[key] = aggregate(world, cfg.n_tok, args.steps, v, max_over_ranks)
    del layer, p, dy, b, ws
    torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """Forward and forward+backward timing of the layer under prescribed load
    skews: bf16, MXFP8 operands (the MXFP8 backward quantises every expert
    GEMM's operands as its forward does), FP8 weights with per-tile scales,
    and the capacity-factor drop mode.  Routing comes from the workload's
    own gate and bias ("bias") or from synthetic fp32 logits through
    moe_route_from_logits (uniform, Zipf s=1, half of the tokens on expert 0)."""
    import torch

    from ragged_grouped_gemm_gb300 import api
    from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_dy, make_layer, skewed_logits
    base = CONFIGS[args.workload]
    peaks = measured_peaks()
    dev = torch.device("cuda", 0)
    p = make_layer(base, dev)
    dy = make_dy(base, dev)
    results = []
    # dropless bf16 and MXFP8, then the capacity-factor (drop) comparison in bf16
    for prec, cap_f in (("bf16", 0.0), ("mxfp8", 0.0), ("fp8w", 0.0), ("bf16", 1.0), ("bf16", 1.25)):
        cfg = base.replace(precision=prec, capacity_factor=cap_f)
        layer = api.MoELayer(cfg, p, train=True, device=dev)
        b, d, ws = layer.buf, layer.desc, layer.ws
        for skew in ("bias", "uniform", "zipf", "half0"):
            lg = None if skew == "bias" else skewed_logits(cfg.n_tok, cfg.n_exp, skew).to(dev)
            zero_bias = torch.zeros(cfg.n_exp, dtype=torch.float32, device=dev) if cfg.use_bias else None

            def fwd():
                if lg is None:
                    return layer.forward(p["x"])
                api.moe_route_from_logits(d, lg, zero_bias, b["topk_idx"], b["topk_w"], b["counts"],
                                          b["offsets_full"] if layer.cap else b["offsets"], ws)
                b["logits"].copy_(lg)        # the router gradient reads the logits the routing used
                layer.x = p["x"]
                if layer.mx:
                    return layer._forward_mx(p["x"])
                layer._permute(p["x"])
                return layer._ffn_combine(p["x"])

            def fwd_bwd():
                fwd()
                layer.backward(dy)

            def timed(fn):
                for _ in range(args.warmup):
                    fn()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    fn()
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1) / args.steps
            ms = timed(fwd)
            ms_fb = timed(fwd_bwd)
            counts = b["counts"].cpu()
            ne = int((counts > 0).sum())
            wb = 3 * ne * cfg.d_ff * cfg.d_model + (3 * cfg.d_ff_shared * cfg.d_model if cfg.n_shared else 0)
            wbytes = wb * (1 + 1 / 32) if prec == "mxfp8" else (wb * (1 + 4 / 128 ** 2) if prec == "fp8w" else 2 * wb)
            results.append({"precision": prec, "capacity_factor": cap_f, "drop_rate": layer.drop_rate(),
                            "skew": skew, "ms_fwd": ms, "tokens_per_s": cfg.n_tok / ms * 1e3,
                            "experts_nonempty": ne, "max_load_over_mean": float(counts.max()) / (cfg.rows / cfg.n_exp),
                            "weight_bytes": wbytes, "weight_stream_gbs": wbytes / ms / 1e6,
                            "weight_stream_frac_of_hbm": wbytes / ms / 1e6 / peaks["hbm_gbs"],
                            "tflops": flops(cfg)["ffn_fwd"] / ms / 1e9, "ms_fwd_bwd": ms_fb,
                            "tokens_per_s_fwd_bwd": cfg.n_tok / ms_fb * 1e3,
                            "tflops_fwd_bwd": (flops(cfg)["ffn_fwd"] + flops(cfg)["ffn_bwd"]) / ms_fb / 1e9})
            assert layer.device_status()[0] == 0
        del layer
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": f"{base.name} forward and forward+backward, steps={args.steps}", "peaks": peaks,
                      "results": results}),
          flush=True)


def call_bytes(cfg) -> dict:
    """Algorithmic HBM bytes of the memory-bound calls of one forward: the
    bytes each must read and write at least, whatever kernels it uses.
    route: x and W_g read, logits, top-K indices and weights, counts and
    offsets written; permute: expert indices and x read, the two maps and
    the permuted rows written (MXFP8: E4M3 codes + one scale byte per 32,
    plus the token-order copy with a shared expert); route_permute (both in
    one call): x and W_g read once, every output of both written; combine:
    the permuted outputs, maps and weights read (+ the shared output), the
    output written."""
    n, d, e, k = cfg.n_tok, cfg.d_model, cfg.n_exp, cfg.top_k
    r = n * k
    q = 1 + 1 / 32
    route = 2 * n * d + 2 * e * d + 4 * n * e + 8 * r + 4 * (2 * e + 1)
    if cfg.precision == "mxfp8":
        permute = 4 * r + 2 * n * d + 8 * r + q * r * d + (q * n * d if cfg.n_shared else 0)
    else:
        permute = 4 * r + 2 * n * d + 8 * r + 2 * r * d
    combine = 2 * r * d + 8 * r + (2 * n * d if cfg.n_shared else 0) + 2 * n * d
    # the fused call reads x and the expert indices only once (x again from L2, the indices it wrote itself)
    route_permute = route + permute - 2 * n * d - 4 * r
    return {"route": route, "permute": permute, "route_permute": route_permute, "combine": combine}


def summarize(res, args, peaks) -> dict:
    """Throughput, per-call times and GB/s, and the roofline of every kind of
    grouped GEMM for one run of run_ours."""
    cfg, per_call, kernels = res["cfg"], res["per_call"], res["kernels"]
    tok_s, ms = res["step"]
    fl = flops(cfg)
    # Tensor-bound kinds are timed inside a step of a few milliseconds, so
    # their roof is the burst bf16 peak (MXFP8: twice it, the nominal
    # fp8/bf16 ratio); the sustained figure is reported beside it.
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    mult, mult_note = (2.0, " x 2 (nominal fp8/bf16 ratio)") if cfg.precision == "mxfp8" else (1.0, "")
    kind_names = {"gate": "router logits GEMM", "ffn_fwd": "forward expert GEMMs (GEMM1 w1|w3+SwiGLU, GEMM2 w2)",
                  "dgrad": "data-gradient GEMMs (through w2 + SwiGLU derivative, through w1|w3)",
                  "wgrad": "weight-gradient GEMMs (dW1, dW3, dW2; fp32 out)"}
    roofs = {}
    for kind, kt in kernels.items():
        if not kt["launches"]:
            continue
        k_fl, k_b = kind_work(cfg, kind, res["nonempty"])
        k_fl, k_b = k_fl * args.steps / kt["launches"], k_b * args.steps / kt["launches"]   # per launch
        k_s = kt["ms_total"] / kt["launches"] / 1e3
        m = 1.0 if kind == "gate" else mult
        kpeak = burst * m
        if k_fl / (kpeak * 1e12) >= k_b / (peaks["hbm_gbs"] * 1e9):
            r = {"bound": "tensor", "achieved": k_fl / k_s / 1e12, "peak": kpeak, "unit": "TFLOP/s",
                 "peak_source": f"{peaks['source']} bf16_tflops (burst)" + (mult_note if m > 1 else ""),
                 "peak_sustained": sustained * m, "frac_of_sustained": k_fl / k_s / 1e12 / (sustained * m)}
        else:
            r = {"bound": "hbm", "achieved": k_b / k_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "peak_source": f"{peaks['source']} hbm_gbs"}
        tkey = kind if cfg.precision == "bf16" else f"{kind}_{cfg.precision}"
        r.update(frac=r["achieved"] / r["peak"], traffic=recorded_traffic(tkey, cfg.name), kernel=kind_names[kind],
                 launches_per_step=kt["launches"] / args.steps, ms_per_launch=k_s * 1e3,
                 share_of_step=kt["ms_total"] / ms, algorithmic_flops=k_fl, algorithmic_bytes=k_b,
                 tflops=k_fl / k_s / 1e12)
        roofs[kind] = r
    cb = call_bytes(cfg)
    per_call_gbs = {c: {"gbs": cb[c] / (per_call[c] / 1e3) / 1e9,
                        "frac_of_hbm": cb[c] / (per_call[c] / 1e3) / 1e9 / peaks["hbm_gbs"],
                        "algorithmic_bytes": cb[c]} for c in cb if c in per_call}
    return {
        "workload": workload_name(cfg), "value": tok_s, "unit": "tokens/s", "ms_per_step": ms / args.steps,
        "fwd_tokens_per_s": res["fwd"][0],
        "grouped_ffn_tflops": fl["ffn_fwd"] / (per_call["grouped_ffn"] / 1e3) / 1e12,
        "backward_tflops": (fl["ffn_bwd"] + fl["router_bwd"]) / (per_call["backward"] / 1e3) / 1e12,
        "per_call_ms": per_call, "per_call_gbs": per_call_gbs, "roofline_by_kind": roofs,
        "e2e": {"value": res["e2e"][0], "unit": "tokens/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]},
        "max_load_over_mean": res["max_load_over_mean"], "clocks": res["clocks"],
        # forward only, no saved activations: GEMM1 rows gathered from x by TMA
        # (no permuted copy of the tokens) against the same forward through x_perm
        "inference_fwd_tokens_per_s": res.get("inference_fwd"),
    } | ({"mxfp8_weight_quantisation": {
        "ms_per_update": res["weight_quant_ms"], "in_value": False,
        "what": "rowwise and columnwise E4M3 codes + E8M0 scales of every expert weight, made once per weight "
                "update (not per forward + backward); amortised over the steps between updates"}}
        if res.get("weight_quant_ms") is not None else {})


# Further configurations timed after the headline one (one GPU only): the
# DeepSeek-V3-shaped layer in bf16 and MXFP8 and the Mixtral-shaped layer in
# MXFP8, each reported with its own roofline and clocks.
SUB_CONFIGS = [("dsv3", "bf16"), ("dsv3", "mxfp8"), ("mixtral", "mxfp8")]


def main():
    args = parse()
    if args.sweep:
        run_sweep(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from ragged_grouped_gemm_gb300.inputs import CONFIGS
    cfg = CONFIGS[args.workload].replace(precision=args.precision)
    tokens_per_step = cfg.n_tok

    if args.impl == "reference":
        if rank != 0:
            return
        sample = args.sample or 64
        n, times = time_oracle(cfg, sample, steps=args.warmup + args.steps)
        t = times[args.warmup:] if len(times) > args.warmup else times
        sec = statistics.mean(t)
        val = n / sec
        cores = os.cpu_count()
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3 * tokens_per_step / n,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic", "config": {"workload": workload_name(cfg), "sample_tokens": n},
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{n} seeded tokens of the {cfg.name} batch, fwd+bwd, numpy fp32"
                                           + ("" if cfg.precision == "bf16" else f", {cfg.precision} oracle")},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, cfg, rank, world, local_rank)
    subs = []
    if world == 1 and not args.no_sub_configs and (args.workload, args.precision) == ("mixtral", "bf16"):
        for wl, prec in SUB_CONFIGS:
            subs.append(run_ours(args, CONFIGS[wl].replace(precision=prec), rank, world, local_rank))
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    peaks = measured_peaks()
    head = summarize(res, args, peaks)
    roofs = head["roofline_by_kind"]
    dominant = max(roofs, key=lambda kk: roofs[kk]["share_of_step"])
    roof = dict(roofs[dominant])
    roof["kind"] = dominant
    dtype = {"bf16": "bf16", "mxfp8": "mxfp8 (e4m3 x e4m3, e8m0 scales per 32)",
             "fp8w": "e4m3 weights (fp32 tile scales) x bf16"}[cfg.precision]
    wbytes = {"bf16": 2, "mxfp8": 1 + 1 / 32, "fp8w": 1}[cfg.precision] * 3 * cfg.n_exp * cfg.d_ff * cfg.d_model
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {"workload": head["workload"],
                   "l2": (f"no flush: the {wbytes / 1e9:.1f} GB of expert weights streamed every step exceed "
                          "the 126 MB L2") if wbytes > 126e6 else
                         (f"no flush: the whole workload ({wbytes / 1e6:.1f} MB of weights) fits in the 126 MB L2; "
                          "a latency-bound case"),
                   "seeds": "x=1 W_g=2 W1=3 W3=4 W2=5 shared=6/7/8 dY=9"},
        "fwd_tokens_per_s": head["fwd_tokens_per_s"],
        "grouped_ffn_tflops": head["grouped_ffn_tflops"],
        "backward_tflops": head["backward_tflops"],
        "per_call_ms": head["per_call_ms"],
        "per_call_gbs": head["per_call_gbs"],
        "inference_fwd_tokens_per_s": head["inference_fwd_tokens_per_s"],
        "roofline": roof,
        "roofline_by_kind": roofs,
        "e2e": head["e2e"],
        "gpu_launches": launches_per_step(cfg) * args.steps,
        "clocks": head["clocks"],
    }
    if "mxfp8_weight_quantisation" in head:
        line["mxfp8_weight_quantisation"] = head["mxfp8_weight_quantisation"]
    if subs:
        line["sub_results"] = [summarize(r, args, peaks) for r in subs]
    if not args.no_cpu_baseline:
        sample = args.sample or 64
        n, times = time_oracle(cfg, sample, steps=1)
        line["cpu_baseline"] = {"value": n / times[0], "unit": "tokens/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{n} seeded tokens of the {cfg.name} batch, fwd+bwd, numpy fp32"
                                           + ("" if cfg.precision == "bf16" else f", {cfg.precision} oracle")}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
