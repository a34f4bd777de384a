#!/usr/bin/env python
"""Benchmark of the MoE-LoRA expert layer: one step = forward + backward of the
whole layer (route, permute, grouped split-LoRA SwiGLU GEMMs, combine, and the
backward with dX, routing-weight and LoRA gradients) on one batch.

Default workload: the Qwen3-30B-A3B-shaped layer (T=4096 tokens, d=2048,
f=768, E=128 experts, top-8, LoRA r=64, alpha=128), synthetic seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the layer on its own
batch (weak scaling, no collective on the data path); the elapsed time is the
maximum over ranks.  Rank 0 prints one JSON line.  ``--impl reference`` times
the CPU oracle (plain NumPy fp64) on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer fwd+bwd tokens/s and TFLOP/s vs BF16 peak; routing GB/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# dram__bytes_read.sum + dram__bytes_write.sum of one launch, from one ncu
# capture, keyed by (kernel, workload) and stamped with the digest of the GEMM
# sources the capture ran (kernel_sources_digest); a figure whose stamp no
# longer matches the sources is stale and reported as null.
NCU_TRAFFIC = {
    ("gate_up", "qwen3_30b_a3b"): {"bytes": 998525696 + 273996800, "sources": "f9d482dfa1eb"},
}
GEMM_SOURCES = ("csrc/gemm.cu", "csrc/ptx.cuh", "csrc/internal.h", "csrc/api.cu")


def kernel_sources_digest():
    """Short digest of the sources that define the GEMM kernels and their
    launches (a captured traffic figure holds for these sources only)."""
    import hashlib
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, "expert_routing_grouped_moe_gb300", rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel, config):
    """(bytes, note): the captured DRAM traffic of one launch, or None with the
    reason when there is no capture of the current kernel sources."""
    rec = NCU_TRAFFIC.get((kernel, config))
    if rec is None:
        return None, "no ncu capture of this kernel and workload"
    if rec["sources"] != kernel_sources_digest():
        return None, "stale: the kernel sources changed since the capture (%s)" % rec["sources"]
    return rec["bytes"], "ncu capture of sources %s" % rec["sources"]


def workload(synth, args):
    """The named layer workload, with T replaced when --tokens is given."""
    cfg = synth.CONFIGS[args.config]
    return synth.scaled(cfg, T=args.tokens) if args.tokens > 0 else cfg


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="qwen3_30b_a3b")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count T (0: the workload's own)")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps (capped)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--probe-steps", type=int, default=100)
    ap.add_argument("--no-route-sweep", action="store_true")
    ap.add_argument("--full-grads", action="store_true",
                    help="also compute the full weight gradients dW_gu, dW_dn each step")
    ap.add_argument("--route-only", action="store_true",
                    help="time only moe_route on the routing sweep points")
    ap.add_argument("--rank-r-tokens", action="store_true",
                    help="the LoRA-A products read the token rows (X, dY) instead of the "
                         "permuted copies")
    ap.add_argument("--sweep", action="store_true",
                    help="time route, permute and combine at every routing-workload point "
                         "(with --route-only: routing alone)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- work model

def layer_counts(cfg, full_grads=False):
    """Algorithmic work of one fwd+bwd step (split-LoRA counts; the dense
    merged work is not counted) and, per kernel launch, its FLOPs and two
    byte counts, each input read once and each output written once:

    * method bytes: every saved intermediate as the single bf16 tensor the
      method's step table sizes (h [N,2f], act [N,f], xa_gu / xa_dn / u / v
      [N,r], dh [N,2f]), weights and rows in bf16, LoRA gradients in fp32;
    * stored bytes: what this build stores -- fp32 h and hi/lo bf16 pairs for
      the intermediates that feed a row reduction, routing-weight-gradient
      partials.

    The roofline is reported on the method bytes; the stored bytes show what
    the precision plan costs.  full_grads adds the full weight gradients."""
    T, d, f, r, k = cfg.T, cfg.d, cfg.f, cfg.r, cfg.k
    N = cfg.rows                                   # routed rows (+ shared rows)
    G = cfg.groups
    hs = 32 * ((f + 15) // 16)                     # fp32 h row: [gate 16 | up 16] chunks
    nparts = 2 * ((f + 191) // 192)                # dw partial slices (at most)
    F_base = 2 * N * d * 2 * f + 2 * N * f * d     # gate_up + down
    F_lora = 2 * N * (d * r + r * 2 * f + f * r + r * d)
    W_gu, W_dn = 2 * G * 2 * f * d, 2 * G * d * f
    A_gu, B_gu, A_dn, B_dn = 2 * G * r * d, 2 * G * 2 * f * r, 2 * G * r * f, 2 * G * d * r
    rows_d = 2 * N * d
    # method sizes (bf16) and stored sizes of the intermediates
    m_r, m_f, m_2f = 2 * N * r, 2 * N * f, 2 * N * 2 * f
    p_r, p_f, p_2f = 4 * N * r, 4 * N * f, 4 * N * 2 * f      # hi/lo pairs
    h32 = 4 * N * hs
    kern = {  # per launch: (flops, method bytes, stored bytes)
        "xa_gu": (2 * N * d * r, rows_d + A_gu + m_r, rows_d + A_gu + p_r),
        "gate_up": (2 * N * d * 2 * f + 2 * N * r * 2 * f,
                    rows_d + W_gu + m_r + B_gu + m_2f + m_f,
                    rows_d + W_gu + p_r + B_gu + h32 + p_f),
        "xa_dn": (2 * N * f * r, m_f + A_dn + m_r, p_f + A_dn + p_r),
        # down reads the high halves of act' and xa_dn (both carry w)
        "down": (2 * N * f * d + 2 * N * r * d, m_f + W_dn + m_r + B_dn + rows_d,
                 2 * N * f + W_dn + 2 * N * r + B_dn + rows_d),
        "u": (2 * N * d * r, rows_d + B_dn + m_r, rows_d + B_dn + p_r),
        "dgrad_dn": (2 * N * d * f + 2 * N * r * f,
                     rows_d + W_dn + m_r + A_dn + m_2f + 8 * N + m_2f + 4 * N,
                     rows_d + W_dn + p_r + A_dn + h32 + 8 * N + 2 * p_f + 4 * N * nparts),
        "v": (2 * N * 2 * f * r, m_2f + B_gu + m_r, p_2f + B_gu + p_r),
        "dgrad_gu": (2 * N * 2 * f * d + 2 * N * r * d, m_2f + W_gu + m_r + A_gu + rows_d,
                     2 * N * 2 * f + W_gu + 2 * N * r + A_gu + rows_d),
        "dB_dn": (2 * N * d * r, rows_d + m_r + 4 * G * d * r, rows_d + p_r + 4 * G * d * r),
        "dA_dn": (2 * N * f * r, m_f + m_r + 4 * G * r * f, p_f + p_r + 4 * G * r * f),
        "dB_gu": (2 * N * 2 * f * r, m_2f + m_r + 4 * G * 2 * f * r,
                  p_2f + p_r + 4 * G * 2 * f * r),
        "dA_gu": (2 * N * d * r, rows_d + m_r + 4 * G * r * d, rows_d + p_r + 4 * G * r * d),
        "route": (0, 4 * T * k + 8 * N + 12 * G, 4 * T * k + 8 * N + 12 * G),
        "permute": (0, 2 * T * d + 2 * N * d + 4 * N, 2 * T * d + 2 * N * d + 4 * N),
        "combine": (0, 2 * N * d + 2 * T * d + 8 * N + 4 * T * k,
                    2 * N * d + 2 * T * d + 8 * N + 4 * T * k),
        "dw_reduce": (0, 4 * N * nparts + 4 * N, 4 * N * nparts + 4 * N),
    }
    F_full = 0
    if full_grads:
        kern["dW_gu"] = (2 * N * 2 * f * d, m_2f + rows_d + 4 * G * 2 * f * d,
                         p_2f + rows_d + 4 * G * 2 * f * d)
        kern["dW_dn"] = (2 * N * d * f, m_f + rows_d + 4 * G * d * f,
                         p_f + rows_d + 4 * G * d * f)
        F_full = 2 * N * 2 * f * d + 2 * N * d * f
    return {"flops": 2 * F_base + 3 * F_lora + F_full, "F_base": F_base, "F_lora": F_lora,
            "F_full": F_full, "kernels": kern, "launches": {"permute": 2, "combine": 2}}


# Kernels the backward runs on the library's second stream, beside the dgrad
# chain.  Their event-timed durations include time queued behind the main
# stream's kernels, so they are not roofline candidates.
AUX_STREAM_KERNELS = ("dB_dn", "dA_dn", "dw_reduce", "dB_gu", "dA_gu", "dW_dn", "dW_gu")


def read_stream_gbs(torch, L, dev, reps=5):
    """Rates at which this GPU streams reads alone, from the library's
    read-stream probe over a 1 GiB buffer (no compute), L2 evicted before each
    call, median of `reps` calls: linear 32 KB bulk copies, and GEMM-operand
    tiles (TMA boxes of 128 rows x 128 bytes, each SM on its own rows).
    Context for read-dominated kernels: the copy peak in MEASURED_PEAKS.json
    mixes reads and writes."""
    x = torch.ones(1 << 29, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for name, pattern in (("linear", L.MOE_PROBE_LINEAR), ("tiles", L.MOE_PROBE_TILES)):
        L.moe_probe_read_stream(x, pattern)
        times = []
        for i in range(reps):
            flush.fill_(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            L.moe_probe_read_stream(x, pattern)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        times.sort()
        out[name] = (1 << 30) / (times[len(times) // 2] / 1e3) / 1e9
    if L.moe_status() != L.MOE_OK:
        raise SystemExit("device status error in the read-stream probe")
    del x, flush
    torch.cuda.empty_cache()
    return out


def kernel_roofline(name, flops, nbytes, dur_s, peaks, stored_bytes=None):
    """Roofline of one launch on the method's bytes: bound = whichever of the
    tensor time (flops / sustained bf16 peak) and the HBM time (bytes / copy
    peak) is longer; achieved is the work of that kind per second.  The
    stored-precision bytes give the fraction this build's own traffic runs
    at, as context."""
    t_tensor = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        ach, peak, unit, bound = flops / dur_s / 1e12, peaks["bf16_tflops_sustained"], \
            "TFLOP/s", "tensor"
    else:
        ach, peak, unit, bound = nbytes / dur_s / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
    out = {"kernel": name, "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
           "frac": ach / peak, "flops_per_launch": flops, "bytes_per_launch": nbytes,
           "bytes_basis": "method (bf16 intermediates)",
           "tensor_frac": flops / dur_s / 1e12 / peaks["bf16_tflops_sustained"],
           "hbm_frac": nbytes / dur_s / 1e9 / peaks["hbm_gbs"]}
    if stored_bytes is not None:
        out["stored_bytes_per_launch"] = stored_bytes
        out["stored_hbm_frac"] = stored_bytes / dur_s / 1e9 / peaks["hbm_gbs"]
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in PEAKS_FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 200 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons, power = [], None, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        loaded = [x for x in sm if mx and x > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- distributed

def dist_setup(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, rank, world, local


def max_over_ranks(torch, dist, value, device):
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_rank, ms_max):
    """Whole-job tokens/s of `world` replicas that each process
    `tokens_per_rank` tokens per step, timed by the slowest rank."""
    return world * tokens_per_rank / (ms_max / 1e3)


def barrier(dist, torch, device):
    if dist is not None:
        if device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- CPU oracle

def oracle_time_per_token(P, X, ids, w, dY, ntok):
    import oracle
    t0 = time.perf_counter()
    oracle.layer_forward(X[:ntok], ids[:ntok], w[:ntok], P)
    oracle.layer_backward(X[:ntok], ids[:ntok], w[:ntok], dY[:ntok], P)
    return (time.perf_counter() - t0) / ntok


def oracle_inputs(cfg, weights, act, ids, w):
    """fp64 copies of the synthetic workload for the oracle (host side)."""
    import numpy as np
    import oracle
    P = oracle.OracleParams.from_arrays(
        {n: t.double().cpu().numpy() for n, t in weights.items()}, s=cfg.scale, E=cfg.E,
        shared=cfg.shared)
    X = act["X"].double().cpu().numpy()
    dY = act["dY"].double().cpu().numpy()
    return P, X, np.ascontiguousarray(ids), np.ascontiguousarray(w), dY


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        nt = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if nt:
            return int(max(nt))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline(cfg, P, X, ids, w, dY, budget_s):
    """The oracle as it stands on a bounded token sample, as tokens/s."""
    tpt = oracle_time_per_token(P, X, ids, w, dY, min(cfg.T, 8))
    ntok = int(max(8, min(cfg.T, budget_s / max(tpt, 1e-9))))
    t0 = time.perf_counter()
    import oracle
    oracle.layer_forward(X[:ntok], ids[:ntok], w[:ntok], P)
    oracle.layer_backward(X[:ntok], ids[:ntok], w[:ntok], dY[:ntok], P)
    dt = time.perf_counter() - t0
    return {"value": ntok / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "oracle fp64 forward+backward of the first %d of %d tokens "
                      "(all %d slots, every expert they route to), %.1f s" % (
                          ntok, cfg.T, cfg.slots, dt)}


# ---------------------------------------------------------------- e2e / sweep

def run_e2e(torch, layer, X, dY, ids, topw, cfg, steps, main):
    """ms per step of forward+backward through the public API, inputs copied
    from pinned host buffers and Y, dX copied back every step."""
    Xh, dYh = X.cpu().pin_memory(), dY.cpu().pin_memory()
    idsh, wh = ids.cpu().pin_memory(), topw.cpu().pin_memory()
    Yh = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
    dXh = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
    dev_in = [(torch.empty_like(X), torch.empty_like(dY), torch.empty_like(ids),
               torch.empty_like(topw)) for _ in range(2)]
    cs = torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    buf_free = [torch.cuda.Event() for _ in range(2)]
    fwd_done, bwd_done, y_out, dx_out = (torch.cuda.Event() for _ in range(4))
    for e in buf_free:
        e.record(main)
    y_out.record(main)
    dx_out.record(main)

    def h2d(i):
        b = i % 2
        cs.wait_event(buf_free[b])
        Xd, dYd, idd, wd = dev_in[b]
        with torch.cuda.stream(cs):
            Xd.copy_(Xh, non_blocking=True)
            idd.copy_(idsh, non_blocking=True)
            wd.copy_(wh, non_blocking=True)
            dYd.copy_(dYh, non_blocking=True)
        in_ready[b].record(cs)

    def step(i):
        b = i % 2
        Xd, dYd, idd, wd = dev_in[b]
        main.wait_event(in_ready[b])
        main.wait_event(y_out)            # the previous Y has left the device
        Y = layer.forward(Xd, idd, wd)
        fwd_done.record(main)
        cs.wait_event(fwd_done)
        with torch.cuda.stream(cs):
            Yh.copy_(Y, non_blocking=True)
        y_out.record(cs)
        main.wait_event(dx_out)
        g = layer.backward(dYd)
        bwd_done.record(main)
        buf_free[b].record(main)
        cs.wait_event(bwd_done)
        with torch.cuda.stream(cs):
            dXh.copy_(g["dX"], non_blocking=True)
        dx_out.record(cs)

    def run(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            step(i)
        main.wait_stream(cs)

    run(3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(main)
    cs.wait_event(e0)
    run(steps)
    e1.record(main)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


DEFAULT_SWEEP_POINTS = ((1 << 20, 128, 8, "uniform"), (1 << 20, 128, 8, "zipf"),
                        (1 << 18, 64, 4, "uniform"))


def routing_sweep(torch, L, synth, dev, peaks, points=DEFAULT_SWEEP_POINTS, d=2048, reps=5,
                  route_only=False):
    """Route, permute and combine throughput (algorithmic GB/s) on points of
    the routing workload: T tokens, E experts, top-k ids (uniform or Zipf),
    bf16 rows of d.  Each call is timed on its own with CUDA events, after a
    write of 256 MB (twice L2) that evicts its inputs from L2; `pipeline` is
    the three calls' bytes over their summed times.  route_only: routing
    alone, with only the id and routing-table buffers allocated."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = []
    for T, E, k, dist in points:
        ids = synth.topk_ids(T, E, k, dist, seed=7, device=dev)
        N = T * k
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        tile_off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        src = torch.empty(N, dtype=torch.int32, device=dev)
        dst = torch.empty(N, dtype=torch.int32, device=dev)
        ws = torch.empty(L.moe_route_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
        calls = {
            "route": (lambda: L.moe_route(ids, E, False, counts, offsets, tile_off, src, dst, ws),
                      4 * T * k + 8 * N + 12 * E),
        }
        if not route_only:
            w = synth.combine_weights(T, k, seed=7, device=dev)
            X = synth.hidden_rows(T, d, seed=7, device=dev)
            Xp = torch.empty(N, d, dtype=torch.bfloat16, device=dev)
            Y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
            calls["permute"] = (lambda: L.moe_permute(X, k, dst, Xp),
                                2 * T * d + 2 * N * d + 4 * N)
            calls["combine"] = (lambda: L.moe_unpermute_combine(Xp, dst, k, False, Y, weights=w),
                                2 * N * d + 2 * T * d + 8 * N + 4 * T * k)
        res = {"T": T, "E": E, "k": k, "dist": dist, "d": d}
        # context: the same routing step written with PyTorch ops, as the pages
        # do it (stable sort of the flattened ids, one bincount, offsets by a
        # cumulative sum, the inverse permutation by a scatter)
        flat = ids.view(-1)

        def torch_route():
            order = torch.argsort(flat, stable=True)
            cnt = torch.bincount(flat, minlength=E)
            offs = torch.cumsum(cnt, 0)
            inv = torch.empty_like(order)
            inv[order] = torch.arange(N, device=dev)
            return offs, inv
        calls_ctx = {"torch_ops_route": (torch_route, 4 * T * k + 8 * N + 12 * E)}
        tot_ms, tot_b = 0.0, 0
        for name, (fn, nbytes) in calls.items():
            fn()
            torch.cuda.synchronize()
            total = 0.0
            for _ in range(reps):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                total += e0.elapsed_time(e1)
            ms = total / reps
            gbs = nbytes / (ms / 1e3) / 1e9
            res[name] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]}
            tot_ms += ms
            tot_b += nbytes
        if not route_only:
            gbs = tot_b / (tot_ms / 1e3) / 1e9
            res["pipeline"] = {"ms": tot_ms, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]}
        for name, (fn, nbytes) in calls_ctx.items():
            fn()
            torch.cuda.synchronize()
            total = 0.0
            for _ in range(reps):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                total += e0.elapsed_time(e1)
            res[name] = {"ms": total / reps,
                         "note": "context, not this library: torch.argsort(stable) + bincount + "
                                 "cumsum + inverse scatter on the same ids"}
        out.append(res)
        calls.clear()
        X = Xp = Y = w = None  # noqa: F841  (free this point's rows before the next)
        torch.cuda.empty_cache()
    if L.moe_status() != L.MOE_OK:
        raise SystemExit("device status error in the routing sweep")
    return out


def run_sweep(args):
    """Every point of the routing workload (T in 1K..1M, E in 8..128, top-2/4/8,
    uniform and Zipf ids): route, permute and combine GB/s, one JSON line."""
    import torch
    from expert_routing_grouped_moe_gb300 import _lib as L, build, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    L.load()
    peaks, src = load_peaks()
    res = routing_sweep(torch, L, synth, dev, peaks, points=synth.ROUTE_SWEEP,
                        reps=max(1, min(args.steps, 5)), route_only=args.route_only)
    return {"metric": "routing GB/s (route%s), every routing-workload point" % (
                "" if args.route_only else ", permute, combine"),
            "unit": "GB/s", "peak": {"hbm_gbs": peaks["hbm_gbs"], "source": src},
            "timing": "CUDA events per call, L2 evicted by a 256 MB write before each, mean of "
                      "%d calls" % max(1, min(args.steps, 5)),
            "routing_sweep": res}


def run_route_only(args):
    """Routing alone on the sweep's large points (the command the routing
    profiles are taken with): small allocations, one JSON line."""
    import torch
    from expert_routing_grouped_moe_gb300 import _lib as L, build, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    L.load()
    res = routing_sweep(torch, L, synth, dev, peaks=load_peaks()[0], reps=args.steps,
                        points=((1 << 20, 128, 8, "uniform"), (1 << 18, 64, 4, "uniform")),
                        route_only=True)
    return {"metric": "routing GB/s (route only)", "unit": "GB/s", "routing_sweep": res}


# ---------------------------------------------------------------- our arm

def config_dict(cfg, args, world):
    """The workload as both arms report it (the same keys and values)."""
    return {"workload": "%s-shaped MoE-LoRA layer fwd+bwd%s%s" % (
                cfg.name, " with full weight gradients" if args.full_grads else "",
                " at T=%d" % cfg.T if args.tokens > 0 else ""),
            "T": cfg.T, "d": cfg.d, "f": cfg.f, "E": cfg.E, "k": cfg.k, "r": cfg.r,
            "alpha": cfg.alpha, "shared_expert": cfg.shared,
            "global_batch_tokens": world * cfg.T, "parallelism": "replicas x%d" % world,
            "l2": "inputs larger than L2 (%.2f GB of expert weights read per pass)" % (
                2 * (cfg.groups * (2 * cfg.f * cfg.d + cfg.d * cfg.f)) / 1e9)}


def run_ours(args):
    import torch
    from expert_routing_grouped_moe_gb300 import (MoELoRALayer,
                                                  _lib as L, build, synth)

    dist, rank, world, local = dist_setup(torch)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the layer has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    L.load()
    cfg = workload(synth, args)
    seed = args.seed + 1000 * rank
    weights = synth.layer_weights(cfg, seed, device=dev)
    act = synth.layer_activations(cfg, seed, device=dev)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
    topw = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    L.moe_router_topk(act["logits"], cfg.k, ids, topw)
    layer = MoELoRALayer(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.r, cfg.alpha, weights,
                         shared_expert=cfg.shared, device=dev, full_grads=args.full_grads,
                         rank_r_tokens=args.rank_r_tokens)
    X, dY = act["X"], act["dY"]
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        layer.step(X, ids, topw, dY)
    torch.cuda.synchronize()
    if L.moe_status() != L.MOE_OK:
        raise SystemExit("device status error after warm-up")

    counts = layer_counts(cfg, full_grads=args.full_grads)
    names = L.kernel_names()

    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(dist, torch, dev)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        layer.step(X, ids, topw, dY)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, torch, dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(torch, dist, ms, dev)
    if L.moe_status() != L.MOE_OK:
        raise SystemExit("device status error in the timed region")

    # per-kernel device times: a separate pass of the same step loop right
    # after the timed region (the probe's events between launches would stop
    # each kernel from overlapping its set-up with the previous one, so the
    # timed steps above carry no probes)
    probe_steps = min(args.steps, args.probe_steps)
    probes = {}
    for n in names:
        if n in ("router_topk",):
            continue
        per = counts["launches"].get(n, 1)
        probes[n] = L.KernelProbe(n, per * probe_steps)
    for _ in range(probe_steps):
        layer.step(X, ids, topw, dY)
    torch.cuda.synchronize()
    kstats = {}
    for n, pr in probes.items():
        ts = pr.times_ms()
        pr.disarm()
        if ts:
            per = counts["launches"].get(n, 1)
            mean = sum(ts) / len(ts)
            kstats[n] = {"ms_per_launch": mean, "launches_per_step": per,
                         "share": mean * per / ms}

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs (X, ids, w, dY) in from pinned host memory and its
    # results (Y, dX) back out; the copies run on a second stream and overlap
    # the neighbouring step's compute (double-buffered device inputs).
    e2e_steps = args.e2e_steps or min(args.steps, 200)
    e2e_ms = run_e2e(torch, layer, X, dY, ids, topw, cfg, e2e_steps, stream)
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, dev)
    h2d = (X.numel() * X.element_size() + dY.numel() * dY.element_size()
           + ids.numel() * ids.element_size() + topw.numel() * topw.element_size())
    d2h = 2 * cfg.T * cfg.d * 2
    barrier(dist, torch, dev)

    route_sweep = routing_sweep(torch, L, synth, dev, peaks=load_peaks()[0]) \
        if (rank == 0 and not args.no_route_sweep) else None

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    read_gbs = read_stream_gbs(torch, L, dev)
    tokens_s = replica_throughput(world, cfg.T, ms_max)
    tflops = world * counts["flops"] / (ms_max / 1e3) / 1e12
    # dominant kernel and its roofline
    # dominant kernel (largest share of the step among the main-stream
    # kernels, whose event-timed durations are their own) and its roofline
    main = [n for n in kstats if n not in AUX_STREAM_KERNELS]
    dom = max(main, key=lambda n: kstats[n]["share"]) if main else None
    roof = None
    if dom is not None:
        fl, nb, sb = counts["kernels"][dom]
        roof = kernel_roofline(dom, fl, nb, kstats[dom]["ms_per_launch"] / 1e3, peaks,
                               stored_bytes=sb)
        # the ncu figure holds for the workload's own T and the captured sources only
        if args.tokens <= 0:
            roof["traffic"], roof["traffic_source"] = ncu_traffic(dom, args.config)
        else:
            roof["traffic"], roof["traffic_source"] = None, "no capture at this T"
        roof["peak_source"] = "%s (%s)" % (peak_src, "bf16 sustained" if roof["bound"] == "tensor"
                                           else "HBM copy")
        if roof["bound"] == "hbm" and read_gbs:
            roof["context"] = {
                "read_stream_gbs": {k: round(v, 1) for k, v in read_gbs.items()},
                "frac_of_read_stream": {k: roof["achieved"] / v for k, v in read_gbs.items()},
                "read_stream_how": "moe_probe_read_stream over 1 GiB, no compute, L2 evicted, "
                                   "median of 5: linear = 32 KB bulk copies, neighbouring SMs "
                                   "on neighbouring chunks; tiles = TMA boxes of 128 rows x "
                                   "128 B, each SM on its own rows (a GEMM operand's pattern)"}
    route = None
    if "route" in kstats:
        rb = counts["kernels"]["route"][1]  # method bytes (= stored: integer tables)
        gbs = rb / (kstats["route"]["ms_per_launch"] / 1e3) / 1e9
        route = {"gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"], "bytes_per_launch": rb}
    kernels = {}
    for n, v in sorted(kstats.items(), key=lambda kv: -kv[1]["share"]):
        fl, nb, sb = counts["kernels"][n]
        rf = kernel_roofline(n, fl, nb, v["ms_per_launch"] / 1e3, peaks, stored_bytes=sb)
        kernels[n] = {"ms": round(v["ms_per_launch"], 5), "share": round(v["share"], 4),
                      "stream": "aux" if n in AUX_STREAM_KERNELS else "main",
                      "bound": rf["bound"], "frac": round(rf["frac"], 3),
                      "stored_hbm_frac": round(rf["stored_hbm_frac"], 3)}
    gemm_ms = sum(v["ms_per_launch"] * v["launches_per_step"] for n, v in kstats.items()
                  if counts["kernels"][n][0] > 0 and n not in AUX_STREAM_KERNELS)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import numpy as np
        P, Xo, ido, wo, dYo = oracle_inputs(cfg, weights, act, ids.cpu().numpy(),
                                            topw.cpu().numpy())
        cpu = cpu_baseline(cfg, P, Xo, ido, wo, dYo, args.cpu_budget_s)
        del P, Xo, dYo, np

    out = {
        "metric": METRIC, "value": tokens_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the layer shape)",
        "config": config_dict(cfg, args, world),
        "tflops": tflops,
        "tflops_frac": tflops / (world * peaks["bf16_tflops_sustained"]),
        "tflops_frac_of": "%s bf16 sustained %.1f TFLOP/s per GPU" % (
            peak_src, peaks["bf16_tflops_sustained"]),
        "gemm_ms_per_step_main_stream": gemm_ms,
        "routing": route,
        "routing_sweep": route_sweep,
        "roofline": roof,
        "kernels": kernels,
        "kernels_note": ("ms = CUDA-event time per launch on the launching stream in a "
                         "separate probe pass; the weight-gradient kernels (stream 'aux') "
                         "run beside the main stream's dgrad chain, so their span includes "
                         "time spent waiting for and sharing SMs, and their frac "
                         "understates the kernel (serialised ncu times are in profiles/)"),
        "cpu_baseline": cpu,
        "e2e": {"value": world * cfg.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * layer.launches_per_step(),
        "clocks": clocks,
    }
    if dist is not None:
        dist.destroy_process_group()
    return out


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle, as it stands, on the host cores; one step = oracle
    fwd+bwd on a token sample sized so the whole run ends within minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import numpy as np
    import oracle
    from expert_routing_grouped_moe_gb300 import synth
    cfg = workload(synth, args)
    weights = synth.layer_weights(cfg, args.seed, device="cpu")
    act = synth.layer_activations(cfg, args.seed, device="cpu")
    ids, w = oracle.router_topk(act["logits"].numpy(), cfg.k)
    P, X, ids, w, dY = oracle_inputs(cfg, weights, act, ids, w)
    budget = 150.0
    tpt = oracle_time_per_token(P, X, ids, w, dY, min(cfg.T, 8))
    ntok = int(max(1, min(cfg.T, budget / (args.steps + args.warmup) / max(tpt, 1e-9))))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        sel = rng.choice(cfg.T, size=ntok, replace=False)
        oracle.layer_forward(X[sel], ids[sel], w[sel], P)
        oracle.layer_backward(X[sel], ids[sel], w[sel], dY[sel], P, full=args.full_grads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sel = rng.choice(cfg.T, size=ntok, replace=False)
        oracle.layer_forward(X[sel], ids[sel], w[sel], P)
        oracle.layer_backward(X[sel], ids[sel], w[sel], dY[sel], P, full=args.full_grads)
    dt = time.perf_counter() - t0
    value = args.steps * ntok / dt
    sample = ("each step: oracle fp64 forward+backward of %d random tokens of the %d-token "
              "batch" % (ntok, cfg.T))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, args, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.sweep:
        out = run_sweep(args)
    elif args.route_only:
        out = run_route_only(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
