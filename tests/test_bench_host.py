"""bench.py's host-side pieces on CPU: the reference arm's JSON line (the
oracle timed on a token sample), the per-kind algorithmic work used for the
roofline, and the launch counts."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("precision", ["bf16", "mxfp8", "fp8w"])
def test_reference_arm_prints_one_contract_line(precision):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--precision", precision, "--steps", "1", "--warmup", "0", "--sample", "16"],
                         capture_output=True, text=True, check=True, cwd=ROOT, timeout=300).stdout
    lines = [x for x in out.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert ("mxfp8" in d["config"]["workload"]) == (precision == "mxfp8")


def test_kind_work_matches_the_flop_count():
    sys.path.insert(0, ROOT)
    import bench
    from ragged_grouped_gemm_gb300.inputs import CONFIGS
    for name in ("mixtral", "dsv3"):
        cfg = CONFIGS[name]
        fl = bench.flops(cfg)
        total = sum(bench.kind_work(cfg, k, cfg.n_exp)[0] for k in ("ffn_fwd", "dgrad", "wgrad"))
        assert total == pytest.approx(fl["ffn_fwd"] + fl["ffn_bwd"])
        # weight gradients write fp32 dW for every expert: at least 3 E D F 4 bytes
        _, b = bench.kind_work(cfg, "wgrad", cfg.n_exp)
        assert b >= 3 * cfg.n_exp * cfg.d_model * cfg.d_ff * 4
        # MXFP8 operands move fewer bytes than bf16 ones
        mx = cfg.replace(precision="mxfp8")
        assert bench.kind_work(mx, "ffn_fwd", cfg.n_exp)[1] < bench.kind_work(cfg, "ffn_fwd", cfg.n_exp)[1]


def test_launch_counts():
    sys.path.insert(0, ROOT)
    import bench
    from ragged_grouped_gemm_gb300.inputs import CONFIGS
    mix, ds = CONFIGS["mixtral"], CONFIGS["dsv3"]
    # forward 4 (routing and permute in one launch; GEMM1, GEMM2, combine)
    # + backward 13 (combine bwd, 5 GEMMs, 3 per-group map kernels, unpermute, router gradient 3)
    assert bench.route_launches(mix) == 1 and bench.fused_dispatch(mix)
    assert bench.launches_per_step(mix) == 4 + 13
    # MXFP8: the fused router, the quantising single-pass permute, GEMM1, GEMM2, combine
    assert not bench.fused_dispatch(mix.replace(precision="mxfp8"))
    # E = 256: dense offsets, logits GEMM (in contraction slices), one kernel for their sum,
    # top-K, histogram and scan; + shared expert (3 forward, 6 backward) + route-bias update
    assert bench.route_launches(ds) == 3
    assert bench.launches_per_step(ds) == 3 + 1 + 3 + 13 + 3 + 6 + 1
    # enough 128-token tiles to fill the GPU: no slices, the same three launches
    assert bench.route_launches(ds.replace(n_tok=65536)) == 3


def test_gpu_arm_json_line_from_fake_timings(monkeypatch, capsys):
    """The GPU arm's JSON assembly (roofline per kind, per-call GB/s, e2e,
    launches, clocks, sub-results), fed with made-up timings instead of a GPU
    run: every contract key is present, the roofline reports the kind with
    the largest share, and tensor-bound kinds divide by the burst bf16 peak
    (twice it for MXFP8 operands)."""
    sys.path.insert(0, ROOT)
    import bench
    from ragged_grouped_gemm_gb300.inputs import CONFIGS

    seen = []

    def fake_run_ours(args, cfg, rank, world, local_rank):
        seen.append((cfg.name, cfg.precision))
        s = args.steps
        kernels = {"gate": {"ms_total": 0.03 * s, "launches": s}, "ffn_fwd": {"ms_total": 1.8 * s, "launches": 2 * s},
                   "dgrad": {"ms_total": 1.9 * s, "launches": 2 * s}, "wgrad": {"ms_total": 2.4 * s, "launches": 3 * s}}
        per_call = {"route": 0.05, "permute": 0.03, "grouped_ffn": 1.86, "combine": 0.02, "backward": 4.4}
        return {"cfg": cfg, "per_call": per_call, "kernels": kernels,
                "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3},
                "nonempty": cfg.n_exp, "max_load_over_mean": 1.1, "inference_fwd": {"gather": 2.2e6, "x_perm": 2.1e6},
                "h2d": 2, "d2h": 1, "step": (640000.0, 6.4 * s),
                "fwd": (2e6, 2.0 * s), "e2e": (600000.0, 6.8 * s),
                "weight_quant_ms": 1.7 if cfg.precision == "mxfp8" else None}

    monkeypatch.setattr(bench, "run_ours", fake_run_ours)
    monkeypatch.setattr(bench, "measured_peaks", lambda: {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                                                          "bf16_tflops_sustained": 1700.0, "source": "measured"})
    for workload in ("mixtral", "tiny"):
        seen.clear()
        monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", workload, "--steps", "3", "--warmup", "3",
                                          "--no-cpu-baseline"])
        bench.main()
        d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                    "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                    "per_call_gbs"):
            assert key in d, key
        r = d["roofline"]
        assert r["kind"] == "wgrad" and r["bound"] in ("tensor", "hbm")
        assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
        assert set(d["roofline_by_kind"]) == {"gate", "ffn_fwd", "dgrad", "wgrad"}
        for kind, rk in d["roofline_by_kind"].items():
            if rk["bound"] == "tensor":
                assert rk["peak"] == pytest.approx(1900.0)
        assert set(d["per_call_gbs"]) == {"route", "permute", "combine"}
        assert d["e2e"]["h2d_bytes_per_step"] == 2 and d["gpu_launches"] == bench.launches_per_step(
            CONFIGS[workload]) * 3
        if workload == "mixtral":
            # the headline is followed by the other configurations, each with its own roofline
            assert seen == [("mixtral", "bf16")] + list(bench.SUB_CONFIGS)
            subs = d["sub_results"]
            assert len(subs) == len(bench.SUB_CONFIGS)
            mx = [x for x in subs if "mxfp8" in x["workload"]]
            # the MXFP8 weights' quantisation is reported beside the step, not in it
            assert mx and all(x["mxfp8_weight_quantisation"]["ms_per_update"] == 1.7 and
                              x["mxfp8_weight_quantisation"]["in_value"] is False for x in mx)
            assert "mxfp8_weight_quantisation" not in d
            assert all("mxfp8_weight_quantisation" not in x for x in subs if "mxfp8" not in x["workload"])
            for x in mx:
                for rk in x["roofline_by_kind"].values():
                    if rk["bound"] == "tensor" and "router" not in rk["kernel"]:
                        assert rk["peak"] == pytest.approx(3800.0)
        else:
            assert seen == [("tiny", "bf16")] and "sub_results" not in d


def test_call_bytes_are_the_algorithmic_minimum():
    sys.path.insert(0, ROOT)
    import bench
    from ragged_grouped_gemm_gb300.inputs import CONFIGS
    m = CONFIGS["mixtral"]
    b = bench.call_bytes(m)
    n, d, r = m.n_tok, m.d_model, m.rows
    # permute reads x once and writes every copy's row; combine reads every copy's row and writes the output
    assert b["permute"] >= 2 * n * d + 2 * r * d
    assert b["combine"] >= 2 * r * d + 2 * n * d
    assert b["route"] >= 2 * n * d
