"""Host-side pieces of bench.py (no GPU): the work model, the CPU-baseline
leg and the reference arm on a small workload."""
import json
import subprocess
import sys
import os

import numpy as np
import pytest
import torch

import bench
import oracle
from expert_routing_grouped_moe_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layer_counts_qwen3_shape():
    cfg = synth.CONFIGS["qwen3_30b_a3b"]
    c = bench.layer_counts(cfg)
    N = 4096 * 8
    F_base = 2 * N * 2048 * 1536 + 2 * N * 768 * 2048
    F_lora = 2 * N * (2048 * 64 + 64 * 1536 + 768 * 64 + 64 * 2048)
    assert c["flops"] == 2 * F_base + 3 * F_lora
    assert abs(c["flops"] / 1e9 - 699.1) < 1.0   # ~699 GFLOP per fwd+bwd step
    fl, nb, sb = c["kernels"]["gate_up"]
    assert fl == 2 * N * 2048 * 1536 + 2 * N * 64 * 1536
    # method bytes: W_gu 805.3 + Xp 134.2 + B_gu 25.2 + xa 4.2 + h (bf16) 100.7
    # + act (bf16) 50.3 = 1119.9 MB, each read or written once
    W_gu = 128 * 1536 * 2048 * 2
    assert nb == W_gu + 2 * N * 2048 + 128 * 1536 * 64 * 2 + 2 * N * 64 + 2 * N * 1536 \
        + 2 * N * 768
    assert abs(nb / 1e6 - 1119.9) < 0.1
    # stored bytes: fp32 h and the hi/lo pairs of xa and act
    assert sb == W_gu + 2 * N * 2048 + 128 * 1536 * 64 * 2 + 4 * N * 64 + 4 * N * 1536 \
        + 4 * N * 768
    assert c["kernels"]["route"][0] == 0 and c["kernels"]["route"][1] > 0
    for name, (_, m, st) in c["kernels"].items():
        assert 0 < m <= st, name


def test_kernel_roofline_picks_the_longer_bound():
    peaks = {"bf16_tflops_sustained": 1000.0, "hbm_gbs": 5000.0}
    # 1 TFLOP and 1 GB: tensor time 1 ms > HBM time 0.2 ms -> tensor-bound
    r = bench.kernel_roofline("k", 1e12, 1e9, 2e-3, peaks)
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-12
    # 1 GFLOP and 10 GB: HBM time 2 ms -> HBM-bound, achieved 10 GB / 4 ms
    r = bench.kernel_roofline("k", 1e9, 1e10, 4e-3, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["achieved"] - 2500.0) < 1e-9


def test_layer_counts_shared_rows():
    cfg = synth.CONFIGS["skewed_shared"]
    c = bench.layer_counts(cfg)
    N = 16384 * 5
    assert c["F_base"] == 2 * N * 2048 * 3072 + 2 * N * 1536 * 2048


def test_cpu_baseline_small():
    cfg = synth.CONFIGS["tiny"]
    wts = synth.layer_weights(cfg, 1)
    act = synth.layer_activations(cfg, 1)
    ids, w = oracle.router_topk(act["logits"].numpy(), cfg.k)
    P, X, ids, w, dY = bench.oracle_inputs(cfg, wts, act, ids, w)
    out = bench.cpu_baseline(cfg, P, X, ids, w, dY, budget_s=0.2)
    assert out["value"] > 0 and out["kind"] == "oracle" and out["cores"] >= 1
    assert "tokens" in out["sample"]


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    # the same config dict as our arm's (so the two lines describe one workload)
    args = bench.parse_args(["--config", "tiny"])
    assert line["config"] == bench.config_dict(synth.CONFIGS["tiny"], args, 1)


def test_ncu_traffic_is_tied_to_the_kernel_sources(monkeypatch):
    digest = bench.kernel_sources_digest()
    assert len(digest) == 12
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("k", "w"), {"bytes": 123, "sources": digest})
    assert bench.ncu_traffic("k", "w")[0] == 123
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("k", "w"), {"bytes": 123, "sources": "0" * 12})
    val, note = bench.ncu_traffic("k", "w")
    assert val is None and "stale" in note
    assert bench.ncu_traffic("nope", "w")[0] is None


def test_sweep_points_cover_the_routing_workload():
    pts = synth.ROUTE_SWEEP
    assert len(pts) == 4 * 4 * 3 * 2
    assert {p[3] for p in pts} == {"uniform", "zipf"}
    assert {(p[0], p[1], p[2], p[3]) for p in bench.DEFAULT_SWEEP_POINTS} <= set(pts)


def test_clock_sampler_parses_lines():
    s = bench.ClockSampler("GPU-abc")
    s.proc = None
    assert s.stop()["sm_mhz"] is None
