#!/usr/bin/env python
"""Benchmark of the fused MoE layer forward on GB300 (tokens/s + roofline).

One step = one moe_forward over one batch: router (logits, TopK, softmax),
dispatch, expert GEMM1 (+GELU), expert GEMM2, combine -- the whole path.
Workload (default): prefill, T=4096 tokens, H=4096, F=14336, E=8, k=2,
seeded synthetic bf16 inputs (x~N(0,1), W_router~N(0,1/H), W1~N(0,1/H),
W2~N(0,1/F)), no capacity limit.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank runs its own batch of T tokens with the
same weights (data-parallel replicas, no collective on the data path);
value = all ranks' tokens / max over ranks of the timed region.
--impl reference times the plain CPU oracle on the host cores instead.

At N = 1 the default run also measures, after the headline line's own
workload, the decode step (weight-stream bound) and the router sweep at
k = 2 (routing bound), each with its own roofline, under "extra_workloads"
(--no-extras skips them).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/sec at 1 GB300 + % of bf16 tensor/HBM roofline"
UNIT = "tokens/s"
WORKLOADS = ("prefill", "decode", "skewed", "skewed_cf1.2", "tiny", "router_k1", "router_k2",
             "router_k4", "router_k8", "prefill_swiglu", "decode_swiglu", "prefill_k1")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture, keyed by workload/kernel and by the sha256 of the kernel
# source it was taken on; reported as null once the source changes.
NCU_TRAFFIC = {
    # prefill workload: dram__bytes_read.sum + dram__bytes_write.sum of one launch
    "prefill/expert_gemm1": {"bytes": 1032561408 + 221230080, "src": "ffn_gemm.cu", "src_sha": "9c589b4d85665278"},
    "prefill/expert_gemm2": {"bytes": 1429054976 + 60358144, "src": "ffn_gemm.cu", "src_sha": "9c589b4d85665278"},
    # router sweep, k = 1: the fused route (router + dispatch in one kernel) of one call
    "router_k1/router+dispatch": {"bytes": 17898496 + 0, "src": ["route_fused.cu", "route_topk.cuh"],
                                  "src_sha": ["a7321e97027ef3df", "ee199279a3609b01"]},
    # decode workload: both GEMMs on the small-batch kernel
    "decode/expert_gemm1": {"bytes": 940161024 + 3989760, "src": "ffn_gemm_small.cu", "src_sha": "ff59fa4c79617713"},
    "decode/expert_gemm2": {"bytes": 941419776 + 5054208, "src": "ffn_gemm_small.cu", "src_sha": "ff59fa4c79617713"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=WORKLOADS, default="prefill")
    p.add_argument("--e2e-steps", type=int, default=100,
                   help="steps of the end-to-end measurement (host buffers, copies in the timed region)")
    p.add_argument("--graph-steps", type=int, default=20,
                   help="forward steps captured per CUDA graph in the timed region")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-stride", type=int, default=16,
                   help="cpu_baseline: the oracle's FFN and combine run on every n-th token")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the decode and router-sweep measurements after the headline")
    return p.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload_cfg(name):
    import moe_synth
    return moe_synth.ALL[name]


def workload_desc(cfg):
    cf = "none" if cfg.capacity_factor is None else cfg.capacity_factor
    return (f"{cfg.name}: T={cfg.T} H={cfg.H} F={cfg.F} E={cfg.E} k={cfg.k} capacity_factor={cf}"
            + (f" bias0={cfg.bias0}" if cfg.bias0 is not None else "")
            + (" experts=SwiGLU" if cfg.act == "swiglu" else ""))


def src_sha(name):
    with open(os.path.join(ROOT, "mixture_experts_layer_12_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(key):
    """DRAM bytes of one launch from NCU_TRAFFIC, or None once a source the
    figure was taken on has changed."""
    tr = NCU_TRAFFIC.get(key)
    if not tr:
        return None
    srcs = tr["src"] if isinstance(tr["src"], list) else [tr["src"]]
    shas = tr["src_sha"] if isinstance(tr["src_sha"], list) else [tr["src_sha"]]
    return tr["bytes"] if all(src_sha(f) == h for f, h in zip(srcs, shas)) else None


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = device.index or 0
        return vis.split(",")[idx] if vis else str(idx)


# ------------------------------------------------------------- multi-rank --

def rank_inputs(cfg, rank: int, world: int) -> dict:
    """Inputs of one data-parallel replica: the layer's weights are shared,
    the tokens x are drawn per rank (seed offset 1000*rank) when world > 1."""
    import moe_synth
    inputs = moe_synth.make_inputs(cfg)
    if world > 1:
        inputs["x"] = moe_synth.make_x(cfg.with_(seed=cfg.seed + 1000 * rank))
    return inputs


def max_over_ranks(value: float, device) -> float:
    """Max of a per-rank float over the process group (identity at N = 1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(tokens_per_rank: int, world: int, steps: int, max_elapsed_ms: float) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_elapsed_ms / 1e3)


# --------------------------------------------------------- work per kernel --

def launched_kernels(shape):
    """The library's kernels per forward step: small batches route and
    dispatch in one launch, and with k = 1 the combine runs inside the second
    expert GEMM, as the library reports for the shape."""
    import mixture_experts_layer_12_gb300 as moe
    in_router, in_gemm = moe.moe_forward_plan(shape)
    return tuple(n for n in moe.KERNEL_NAMES
                 if not (in_router and n == "dispatch") and not (in_gemm and n == "combine"))


FUSED_INTO = {"dispatch": "router", "combine": "expert_gemm2"}


def kernel_work(cfg, n_rows, experts_hit):
    """Algorithmic FLOPs and bytes of one launch of each kernel."""
    T, H, F, E, k = cfg.T, cfg.H, cfg.F, cfg.E, cfg.k
    F1 = 2 * F if getattr(cfg, "act", "gelu") == "swiglu" else F  # W1 columns (gate | up)
    return {
        "router": dict(flops=2.0 * T * H * E, bytes=2.0 * T * H + 2.0 * H * E + 8.0 * T * k),
        "dispatch": dict(flops=0.0, bytes=4.0 * T * k * 3 + 8.0 * E),
        "permute": dict(flops=0.0, bytes=4.0 * n_rows * H + 4.0 * n_rows),
        "expert_gemm1": dict(flops=2.0 * n_rows * H * F1,
                             bytes=2.0 * experts_hit * H * F1 + 2.0 * n_rows * H + 2.0 * n_rows * F),
        "expert_gemm2": dict(flops=2.0 * n_rows * F * H,
                             bytes=2.0 * experts_hit * F * H + 2.0 * n_rows * F + 2.0 * n_rows * H),
        "combine": dict(flops=2.0 * n_rows * H, bytes=2.0 * n_rows * H + 2.0 * T * H + 8.0 * T * k),
    }


# ---------------------------------------------------------------- rooflines --

# A timed region shorter than this, with no power-cap throttling seen in it,
# runs at burst clocks: its GEMMs are measured against the burst bf16 peak.
SUSTAINED_REGION_MS = 1000.0


def tensor_peak(peaks, region_ms, clocks):
    """(peak TFLOP/s, kind) for a contraction timed over `region_ms` with the
    sampled `clocks`: the burst figure for a short region at full clocks, the
    sustained one for a region of a second or more, or one whose clock the
    power cap held down (median below 95% of the maximum with sw_power_cap
    seen; a momentary cap flag at full clock is still a burst)."""
    capped = (bool(clocks) and "sw_power_cap" in clocks.get("reasons", [])
              and clocks.get("sm_mhz", 0.0) < 0.95 * (clocks.get("sm_max_mhz") or 0.0))
    if region_ms >= SUSTAINED_REGION_MS or capped:
        return peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]), "sustained"
    return peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]), "burst"


def roofline(work, ms, peaks, peak_src, region_ms, clocks, name):
    """The roofline object of one kernel: tensor-bound when its arithmetic
    intensity exceeds the ridge of the measured peaks, HBM-bound otherwise."""
    ridge = (peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) * 1e12 /
             (peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]) * 1e9))
    if work["flops"] / max(work["bytes"], 1.0) > ridge:
        ach = work["flops"] / (ms * 1e-3) / 1e12
        peak, kind = tensor_peak(peaks, region_ms, clocks)
        burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "peak_kind": f"bf16 dense, {kind} ({peak_src}): timed region {region_ms:.0f} ms",
                "frac_of_burst": round(ach / burst, 4), "frac_of_sustained": round(ach / sus, 4),
                "kernel": name, "flops_per_launch": work["flops"]}
    ach = work["bytes"] / (ms * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(ach / peak, 4), "peak_kind": f"HBM copy ({peak_src})",
            "kernel": name, "bytes_per_launch": work["bytes"]}


# ------------------------------------------------------------ cpu baseline --

def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def oracle_step(inputs, cfg, rows):
    """The oracle as it stands on one batch of the workload: routing and
    dispatch (capacity included) for all T tokens, then the expert FFN and
    combine for the tokens in `rows` (tokens are independent once routed and
    dispatched).  Returns (seconds of routing + dispatch, seconds of FFN +
    combine)."""
    import oracle
    t0 = time.perf_counter()
    logits, ids, _, w = oracle.route(inputs["x"], inputs["w_router"], cfg.k, bias=inputs["bias"])
    _, _, _, slot = oracle.dispatch(ids, cfg.E, cfg.capacity_factor)
    t1 = time.perf_counter()
    if rows and cfg.has_ffn:
        oracle.combine_rows(inputs["x"], inputs["w1"], inputs["w2"], ids, w, slot, rows,
                            act=cfg.act)
    return t1 - t0, time.perf_counter() - t1


def cpu_baseline(inputs, cfg, stride):
    """Oracle-equivalent full time of one batch: routing + dispatch of all T
    tokens, plus the FFN and combine of every `stride`-th token scaled by
    T / (tokens computed)."""
    import oracle
    oracle.build()
    rows = list(range(0, cfg.T, stride)) if cfg.has_ffn else []
    t_route, t_ffn = oracle_step(inputs, cfg, rows)
    full = t_route + (t_ffn * cfg.T / len(rows) if rows else 0.0)
    what = (f"routing + dispatch of all {cfg.T} tokens ({t_route:.2f} s)"
            + (f" + {cfg.T / len(rows):.0f} x FFN and combine of every {stride}-th token "
               f"({len(rows)} tokens, {t_ffn:.2f} s)" if rows else ""))
    return {"value": cfg.T / full, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"oracle-equivalent full time {full:.2f} s: {what}",
            "cpu": cpu_model(), "nproc": os.cpu_count()}


# --------------------------------------------------------------- reference --

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    import moe_synth
    oracle.build()
    cfg = workload_cfg(args.workload)
    inputs = moe_synth.make_inputs(cfg)
    # each step: routing + dispatch of all T tokens and the FFN of a strided
    # token sample, sized so that warm-up + steps take about 90 s
    n_steps = max(1, args.warmup + args.steps)
    probe = list(range(0, cfg.T, max(1, cfg.T // 4)))[:4] if cfg.has_ffn else []
    t_route, t_probe = oracle_step(inputs, cfg, probe)
    per_token = t_probe / len(probe) if probe else 0.0
    budget = max(0.0, 90.0 / n_steps - t_route)
    n_ffn = 0
    if cfg.has_ffn:
        n_ffn = int(max(1, min(cfg.T // 16 or 1, budget / max(per_token, 1e-9))))
    stride = max(1, cfg.T // n_ffn) if n_ffn else 0
    full_times = []
    for i in range(n_steps):
        rows = list(range((i * 7) % stride, cfg.T, stride))[:n_ffn] if n_ffn else []
        tr, tf = oracle_step(inputs, cfg, rows)
        if i >= args.warmup:
            full_times.append(tr + (tf * cfg.T / len(rows) if rows else 0.0))
    elapsed = sum(full_times)
    value = cfg.T * len(full_times) / elapsed
    sample = (f"per step: routing + dispatch of all {cfg.T} tokens"
              + (f", FFN and combine of {n_ffn} tokens (stride {stride}) scaled to all {cfg.T}"
                 if n_ffn else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * elapsed / max(1, len(full_times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "ffn_tokens_per_step": n_ffn,
                   "parallelism": "host cores (OpenMP over tokens)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample, "cpu": cpu_model(),
                         "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- ours --

def measure_route(args, cfg, device, with_cpu=True):
    """Router sweep: one step = moe_route (router + dispatch) over T tokens.
    Rotates through enough copies of x that the set exceeds L2."""
    import torch
    import mixture_experts_layer_12_gb300 as moe
    import moe_synth
    inputs = moe_synth.make_inputs(cfg, with_ffn=False)
    x0 = inputs["x"].to(device)
    copies = max(2, int(4 * 129e6 // (x0.numel() * 2)) + 1)
    xs = [x0] + [x0.roll(i, dims=1).contiguous() for i in range(1, copies)]
    wr = inputs["w_router"].to(device)
    s = moe.make_shape(cfg.T, cfg.H, 8, cfg.E, cfg.k, cfg.capacity_factor)
    r = moe.alloc_routing(cfg.T, cfg.E, cfg.k, device)
    ws = moe.alloc_route_workspace(s, device)
    stream = torch.cuda.current_stream(device)
    for i in range(max(3, args.warmup)):
        moe.moe_route(s, xs[i % copies], wr, None, r.ids, r.weights, r.counts, r.offsets, r.perm,
                      r.slot, ws, stream)
    torch.cuda.synchronize(device)
    # one CUDA graph holds one pass over all x copies; the timed region
    # replays it, so host launch overhead does not enter the device time
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        for i in range(copies):
            moe.moe_route(s, xs[i], wr, None, r.ids, r.weights, r.counts, r.offsets, r.perm,
                          r.slot, ws)
    torch.cuda.synchronize(device)
    graph.replay()
    torch.cuda.synchronize(device)
    # at least three replays back to back, so that one replay's launch
    # latency does not sit in the per-route time of a short run
    reps = max(3, args.steps // copies)
    K = reps * copies
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    clocks = ClockSampler(gpu_id_for(device))
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(device)
    ev[0].record(stream)
    for _ in range(reps):
        graph.replay()
    ev[1].record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    if moe.moe_get_device_status(ws, stream) != 0:
        raise RuntimeError("device status set during the timed region")
    elapsed = ev[0].elapsed_time(ev[1])
    ms = elapsed / K
    # end to end through the public API with host buffers: H2D of x, the
    # routing, D2H of ids and gate weights, every step, inside the timed region
    E2E = max(1, args.e2e_steps)
    x_host = inputs["x"].pin_memory()
    ids_host = torch.empty(cfg.T, cfg.k, dtype=torch.int32).pin_memory()
    w_host = torch.empty(cfg.T, cfg.k, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(x0)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(3 + E2E):
        if i == 3:
            torch.cuda.synchronize(device)
            e0.record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        moe.moe_route(s, x_dev, wr, None, r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot,
                      ws, stream)
        ids_host.copy_(r.ids, non_blocking=True)
        w_host.copy_(r.weights, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = e0.elapsed_time(e1)
    e2e = {"value": cfg.T * E2E / (e2e_ms * 1e-3), "unit": UNIT,
           "h2d_bytes_per_step": cfg.T * cfg.H * 2, "d2h_bytes_per_step": cfg.T * cfg.k * 8,
           "steps": E2E}

    peaks, src = load_peaks()
    w = kernel_work(cfg, cfg.T * cfg.k, 0)
    route_work = {"flops": w["router"]["flops"],
                  "bytes": w["router"]["bytes"] + w["dispatch"]["bytes"]}
    roof = roofline(route_work, ms, peaks, src, elapsed, clk, "route (router + dispatch)")
    roof["traffic"] = ncu_traffic(f"{cfg.name}/router+dispatch")
    return {
        "metric": METRIC, "value": cfg.T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "step": "moe_route (router + dispatch)",
                   "l2": f"{copies} rotating copies of x ({copies * x0.numel() * 2 / 1e6:.0f} MB > L2)"},
        "gpu_launches": route_launches(s) * K,
        "roofline": roof,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": (cpu_baseline(inputs, cfg, args.cpu_stride)
                         if with_cpu and not args.no_cpu_baseline else None),
    }


def route_launches(shape):
    """Kernels one moe_route call launches: the status clear, the W_router
    padding when E % 8 != 0, the router, and the dispatch unless the router
    does it."""
    import mixture_experts_layer_12_gb300 as moe
    in_router, _ = moe.moe_forward_plan(shape)
    return 2 + (0 if in_router else 1) + (1 if shape.E % 8 else 0)


def measure_forward(args, cfg, device, world=1, rank=0, with_cpu=True):
    """One step = one moe_forward over T tokens (every kernel of the layer)."""
    import torch
    import torch.distributed as dist
    import mixture_experts_layer_12_gb300 as moe

    inputs = rank_inputs(cfg, rank, world)
    dev = {k: (None if v is None else v.to(device)) for k, v in inputs.items()}
    layer = moe.MoELayer(dev["w_router"], dev["w1"], dev["w2"], cfg.k, bias=dev["bias"],
                         capacity_factor=cfg.capacity_factor, act=cfg.act)
    x = dev["x"]
    stream = torch.cuda.current_stream(device)

    def step(events=None):
        # stream=None: the binding uses torch's current stream (the capture
        # stream while a CUDA graph is being captured)
        layer._ensure(cfg.T, device)
        r = layer.routing
        if events is None:
            moe.moe_forward(layer.shape, x, layer.w_router, layer.bias, layer.w1, layer.w2, layer.y,
                            r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, layer.ws)
        else:
            moe.moe_forward_profiled(layer.shape, x, layer.w_router, layer.bias, layer.w1, layer.w2,
                                     layer.y, r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot,
                                     layer.ws, events)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    if moe.moe_get_device_status(layer.ws, stream) != 0:
        raise RuntimeError("device status set during warm-up")

    # The timed steps replay a CUDA graph of R consecutive forward steps, so
    # host launch overhead does not enter the device time.  A second graph of
    # the same steps with the library's per-kernel events (which sit between
    # the kernels and so turn off their overlapped launch) gives the
    # per-kernel split; it is replayed after the timed region.
    R = max(1, min(args.steps, args.graph_steps))
    reps = max(1, args.steps // R)
    K = R * reps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(moe.KERNEL_NAMES) + 1)]
           for _ in range(R)]
    for row in evs:  # materialise the event handles before capture
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    graph_prof = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        for i in range(R):
            step()
    with torch.cuda.graph(graph_prof, stream=cap):
        for i in range(R):
            step(evs[i])
    torch.cuda.synchronize(device)
    for _ in range(2):  # warm replays
        graph.replay()
    torch.cuda.synchronize(device)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    clocks = ClockSampler(gpu_id_for(device))
    clocks.start()
    time.sleep(0.3)  # let the sampler come up
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(device)
    t_start.record(stream)
    for _ in range(reps):
        graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    if moe.moe_get_device_status(layer.ws, stream) != 0:
        raise RuntimeError("device status set during the timed region")

    elapsed_ms = max_over_ranks(elapsed_ms, device)
    ms_per_step = elapsed_ms / K
    value = whole_job_throughput(cfg.T, world, K, elapsed_ms)

    # per-kernel device time: mean over the R steps of the profiled graph's
    # last replay (kernels run back to back, no overlapped launch), after as
    # many replays as the timed region so both see the same sustained clocks
    for _ in range(reps):
        graph_prof.replay()
    torch.cuda.synchronize(device)
    if moe.moe_get_device_status(layer.ws, stream) != 0:
        raise RuntimeError("device status set during the profiled replays")
    names = moe.KERNEL_NAMES
    per_kernel = {n: statistics.fmean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(R))
                  for j, n in enumerate(names)}
    counts = layer.routing.counts.cpu()
    n_rows = int(counts.sum().item())
    experts_hit = int((counts > 0).sum().item())
    work = kernel_work(cfg, n_rows, experts_hit)

    peaks, peak_src = load_peaks()
    dominant = max(per_kernel, key=per_kernel.get)
    kernels = {}
    launched = launched_kernels(layer.shape)
    for n in names:
        ms = per_kernel[n]
        if n not in launched:  # this step runs inside another kernel
            kernels[n] = {"ms": round(ms, 5), "fused_into": FUSED_INTO[n]}
            continue
        kernels[n] = {"ms": round(ms, 5), "share": round(ms / sum(per_kernel.values()), 4),
                      "tflops": round(work[n]["flops"] / (ms * 1e-3) / 1e12, 2),
                      "gbs": round(work[n]["bytes"] / (ms * 1e-3) / 1e9, 1)}
    roof = roofline(work[dominant], per_kernel[dominant], peaks, peak_src, elapsed_ms, clk,
                    dominant)
    roof["traffic"] = ncu_traffic(f"{cfg.name}/{dominant}")

    # end to end through the public API with host buffers: H2D of x, the
    # forward, D2H of y, every step, inside the timed region.  The headline
    # runs the steps through HostPipeline (the next step's x goes up and the
    # previous y comes down while a step computes); `serial_value` is the
    # same with each step's copies and forward back to back.
    from mixture_experts_layer_12_gb300.host_pipeline import HostPipeline
    E2E = max(1, args.e2e_steps)
    x_hosts = [inputs["x"].pin_memory(), inputs["x"].roll(1, dims=0).pin_memory()]
    y_hosts = [torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    r = layer.routing
    x_dev = torch.empty_like(x)
    for i in range(3 + E2E):
        if i == 3:
            torch.cuda.synchronize(device)
            e0.record(stream)
        x_dev.copy_(x_hosts[i % 2], non_blocking=True)
        moe.moe_forward(layer.shape, x_dev, layer.w_router, layer.bias, layer.w1, layer.w2, layer.y,
                        r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, layer.ws, stream)
        y_hosts[i % 2].copy_(layer.y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    serial_ms = max_over_ranks(e0.elapsed_time(e1), device)

    pipe = HostPipeline(layer, cfg.T, device, graphs=True)
    pipe.run(x_hosts * 2, y_hosts * 2, stream)  # warm-up
    torch.cuda.synchronize(device)
    e0.record(stream)
    pipe.run([x_hosts[i % 2] for i in range(E2E)], [y_hosts[i % 2] for i in range(E2E)], stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    if moe.moe_get_device_status(layer.ws, stream) != 0:
        raise RuntimeError("device status set during the end-to-end steps")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), device)
    e2e = {"value": whole_job_throughput(cfg.T, world, E2E, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": cfg.T * cfg.H * 2, "d2h_bytes_per_step": cfg.T * cfg.H * 2,
           "steps": E2E, "overlap": "copies of neighbouring steps overlap the forward "
                                     "(HostPipeline: two device slots, a CUDA graph of the forward per slot)",
           "serial_value": whole_job_throughput(cfg.T, world, E2E, serial_ms)}

    cpu = None
    if with_cpu and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inputs, cfg, args.cpu_stride)

    # free the layer's device memory before the next workload is measured
    del layer, dev, x, x_dev, graph, graph_prof, pipe
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "tokens_per_gpu": cfg.T,
                   "parallelism": f"replicas x{world} (token data-parallel, no collective)",
                   "kept_rows": n_rows, "experts_hit": experts_hit,
                   "timing": f"CUDA events around {reps} replays of a CUDA graph of {R} forward steps "
                             f"({elapsed_ms:.1f} ms); per-kernel times from a second graph of the "
                             "same steps with events between the kernels",
                   "per_kernel_sum_ms": round(sum(per_kernel.values()), 5),
                   "l2": "inputs larger than L2: every step streams all expert weights "
                         f"({2 * (3 if cfg.act == 'swiglu' else 2) * cfg.E * cfg.H * cfg.F / 1e9:.2f} GB)"},
        # + the status clear that opens each call (+ the W_router padding when E % 8 != 0)
        "gpu_launches": (len(launched) + 1 + (1 if cfg.E % 8 else 0)) * K,
        "roofline": roof,
        "kernels": kernels,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }


def measure(args, cfg, device, world=1, rank=0, with_cpu=True):
    if cfg.has_ffn:
        return measure_forward(args, cfg, device, world, rank, with_cpu)
    return measure_route(args, cfg, device, with_cpu)


EXTRA_WORKLOADS = ("decode", "router_k2")


def extra_summary(line):
    """The parts of a workload's line that the headline line carries for it."""
    keep = ("value", "unit", "ms_per_step", "steps", "roofline", "clocks", "e2e", "cpu_baseline",
            "gpu_launches")
    out = {k: line[k] for k in keep if k in line}
    out["workload"] = line["config"]["workload"]
    if "kernels" in line:
        out["kernels"] = line["kernels"]
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)

    from mixture_experts_layer_12_gb300 import build as moe_build
    moe_build.build()

    cfg = workload_cfg(args.workload)
    if not cfg.has_ffn and world > 1:
        raise SystemExit("router-only workloads run on one GPU")
    line = measure(args, cfg, device, world, rank)
    if world == 1 and not args.no_extras and args.workload == "prefill":
        line["extra_workloads"] = {name: extra_summary(measure(args, workload_cfg(name), device))
                                   for name in EXTRA_WORKLOADS}
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
