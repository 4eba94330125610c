"""Benchmark of the routed MXFP4 MoE layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]
                    [--workload all|decode1|decode64|prefill4096|stack4] [--tokens-per-step M]
                    [--eager] [--no-cpu-baseline] [--experts N] [--f F] [stack4 options]

Default (--workload all): one Kimi K3-shaped MoE layer (d=7168, f=1536, E=896, k=16).
  headline  decode1: single-token decode, M=1000 seeded tokens per step run back to back as
            T=1 layer calls.  A step is one pass of the whole hot path (router, top-k,
            bucketing, expert FFNs, combine) over those tokens.  The 15.7 GB expert pool is far
            larger than L2, so each token streams its 16 experts from HBM (the 25.7 MB router
            stays L2-resident across tokens, as it would in a real decode loop).
  configs   decode64: the same layer, M tokens per step in T=64 calls (batched decode);
            prefill4096: a second layer with a +2.0 selection bias on 32 experts, one T=4096
            call per step (tensor-core grouped GEMM path).
Every workload reports tokens/s with inputs resident, the dominant kernel's roofline from an
event-timed pass, e2e through the host-buffer C entry point (k3moe_layer_forward_host), and the
oracle timed on the host cores at all threads and at one thread.  The decode workloads' timed
steps replay the step's layer calls as one CUDA graph captured by the library
(k3moe_graph_create); the eager steps are timed beside them (--eager: eager only).

--workload stack4: four stacked K3 layers in cache mode (pinned host pool, device slots) with
--budget-gb, --miss-path copy-engine|zero-copy, --device-lru and --prefetch none|trace|router;
reports the cache statistics and an LRU / Belady MIN / random replacement study of the same trace.
--experts N and --f F give small cases with the same per-call work for profiler captures.

Prints one JSON line.  With --gpus N > 1 (launched by torchrun) every rank runs an
independent replica of the layer (the layer has no cross-GPU step on one node here);
value = tokens of all ranks / max rank time.

--impl reference times the CPU oracle (plain fp64 C, this repository's oracle/) on the
host cores, on a bounded sample of the single-token decode workload.
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

import numpy as np  # noqa: E402

METRIC = "MoE-layer tokens/s and MXFP4 weight GB/s as % of B300 HBM peak (T=1/64/4096)"
D, F, E, K = 7168, 1536, 896, 16
SEED = 2026
EXPERT_BYTES = 17_547_264
GATEUP_BYTES = 11_698_176     # gate + up region of one expert
DOWN_BYTES = 5_849_088
ROUTER_BYTES = E * D * 4

WORKLOADS = {
    "decode1": dict(T=1, desc="K3 MoE layer, single-token decode: d=7168 f=1536 E=896 k=16, T=1 per call"),
    "decode64": dict(T=64, desc="K3 MoE layer, batched decode: d=7168 f=1536 E=896 k=16, T=64 per call"),
    "prefill4096": dict(T=4096, desc="K3 MoE layer, prefill: d=7168 f=1536 E=896 k=16, T=4096, +2.0 bias on 32 experts"),
    "stack4": dict(T=1, desc="4 stacked K3 MoE layers (d=7168 f=1536 E=896 k=16; between them r=bf16(r+y), "
                             "next input RMSNorm(r)), "
                             "T=1 decode, 62.9 GB expert pool in pinned host memory behind a device LRU cache"),
}


L2_NOTE = {
    "decode1": "inputs larger than L2: 15.7 GB expert pool streamed from HBM (16 experts, 281 MB per call); "
               "router L2-resident",
    "decode64": "inputs larger than L2: about 620 experts (10.9 GB) streamed per call; router L2-resident",
    "prefill4096": "inputs larger than L2: 561 MB of hot experts, 58.7 MB of tokens and 1.9 GB of per-pick "
                   "activations and outputs per call",
}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def _set_ffn_width(f):
    """Expert sizes for an FFN width other than K3's (profiling cases): 17/32 bytes per weight."""
    global F, EXPERT_BYTES, GATEUP_BYTES, DOWN_BYTES
    if f <= 0 or f % 128:
        raise SystemExit("--f must be a positive multiple of 128")
    F = f
    DOWN_BYTES = f * D * 17 // 32
    GATEUP_BYTES = 2 * DOWN_BYTES
    EXPERT_BYTES = 3 * DOWN_BYTES


def _profiling_case(args):
    parts = []
    if args.experts != E:
        parts.append(f"only {args.experts} experts resident")
    if args.f != 1536:
        parts.append(f"f={args.f}")
    return f" [profiling case: {', '.join(parts)}]" if parts else ""


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return j.get("hbm_gbs", 6400.0), j.get("bf16_tflops", 1800.0), "measured"
    return 6400.0, 1800.0, "fallback"


def _bf16_sustained():
    """The sustained (seconds-long, power-capped) bf16 rate, for work timed inside long steps."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh).get("bf16_tflops_sustained", 1400.0), "measured"
    return 1400.0, "fallback"


NOMINAL_HBM_GBS = 8000.0  # the nominal HBM figure the layer's throughput target is stated against


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _source_hash(rel: str) -> str:
    with open(os.path.join(ROOT, rel), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def _traffic_from_profile(kernel_file: str, summary: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as fh:
        for ln in fh:
            if ":" in ln and not ln.startswith("#"):
                a, b = ln.split(":", 1)
                kv[a.strip()] = b.strip()
    if kv.get("source_sha256_16") != _source_hash(kernel_file):
        return None
    try:
        return int(float(kv["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ replica aggregation ---

def job_throughput(units_per_rank: float, ms_rank: float, pg=None, device: str = "cuda"):
    """Whole-job rate over replicas: every rank processed units_per_rank in ms_rank; the job
    took as long as its slowest rank.  Returns (units of all ranks per second, max ms)."""
    ms = ms_rank
    ws = 1
    if pg is not None:
        import torch
        ws = pg.get_world_size()
        t = torch.tensor([ms_rank], dtype=torch.float64, device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    return units_per_rank * ws / (ms / 1e3), ms


def job_rate_min(rate_rank: float, pg=None, device: str = "cuda") -> float:
    """Whole-job rate when each rank measured its own rate: the slowest rank's rate x ranks."""
    if pg is None:
        return rate_rank
    import torch
    t = torch.tensor([rate_rank], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MIN)
    return float(t.item()) * pg.get_world_size()


# --------------------------------------------------------------------------- b300 arm ---

def build_layer(torch, k3, T_max, bias=None, n_exp=E):
    import synth
    nb, sb = synth.expert_bytes(D, F)
    dn = torch.empty(n_exp * nb, dtype=torch.uint8, device="cuda")
    ds = torch.empty(n_exp * sb, dtype=torch.uint8, device="cuda")
    synth.experts_to_device(SEED, 0, 0, n_exp, D, F, dn.data_ptr(), ds.data_ptr())
    Wr = torch.from_numpy(synth.router_weights(SEED, 0, n_exp, D)).cuda()
    b = None if bias is None else torch.from_numpy(bias).cuda()
    layer = k3.k3moe_pack_experts(k3.dims(D, F, n_exp, K, T_max), dn, ds, 1, Wr, b)
    del dn, ds
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layer


def _combine_gbs(prof, T):
    """The combine kernel's HBM rate: T*k per-pick fp32 rows read, T fp32 rows of y written."""
    ms, n = prof["combine"]
    return round((T * K * D * 4 + T * D * 4) / (ms / n / 1e3) / 1e9, 1) if n else None


def _roofline(prof, T, distinct_per_call, hbm_peak, bf16_peak, peak_kind):
    """Roofline of the dominant kernel from the event-timed pass: the gate/up GEMM (tensor
    bound) on the tensor-core path, the gate/up streaming kernel (HBM bound) otherwise."""
    if prof["gemm_gu"][1]:
        gu_ms, gu_n = prof["gemm_gu"]
        flops = 4.0 * F * D * T * K  # 4*f*d flops per pick (gate and up)
        achieved = flops / (gu_ms / gu_n / 1e3) / 1e12
        dn_ms, dn_n = prof["gemm_dn"]
        return {"bound": "tensor", "kernel": "gemm_kernel<gate/up> (tcgen05, fp16 in, fp32 TMEM accumulate)",
                "achieved": round(achieved, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": round(achieved / bf16_peak, 4),
                "peak_kind": f"{peak_kind} (cuBLAS bf16 dense, burst; fp16 dense has the same rate)",
                "algorithmic_flops_per_launch": flops,
                "traffic": _traffic_from_profile("mxfp4_routed_expert_06_b300/csrc/gemm_tc.cu",
                                                 "gemm_gu_prefill_k3_t4096.txt") if T == 4096 else None,
                "down_gemm_tflops": round(2.0 * F * D * T * K / (dn_ms / dn_n / 1e3) / 1e12, 1),
                "combine_kernel_gbs": _combine_gbs(prof, T)}
    gu_ms, gu_n = prof["gateup"]
    gu_bytes = distinct_per_call * GATEUP_BYTES  # each active expert's gate/up bytes once per call
    achieved = gu_bytes / (gu_ms / gu_n / 1e3) / 1e9 if gu_n else None
    summary = {1: "gateup_decode_k3_t1.txt", 64: "gateup_decode_k3_t64.txt"}.get(T)
    traffic = _traffic_from_profile("mxfp4_routed_expert_06_b300/csrc/decode_ffn.cu", summary) if summary else None
    dn_ms, dn_n = prof["down"]
    return {"bound": "hbm", "kernel": "gateup_kernel (gate/up + SwiGLU, register decode)",
            "achieved": None if achieved is None else round(achieved, 1),
            "peak": hbm_peak, "unit": "GB/s",
            "frac": None if achieved is None else round(achieved / hbm_peak, 4),
            "peak_kind": f"{peak_kind} (HBM copy peak)",
            "algorithmic_bytes_per_launch": int(gu_bytes), "traffic": traffic,
            "down_kernel_gbs": round(distinct_per_call * DOWN_BYTES / (dn_ms / dn_n / 1e3) / 1e9, 1) if dn_n else None,
            "combine_kernel_gbs": _combine_gbs(prof, T)}


def measure(torch, k3, layer, T, calls, xs, args, pg, rank, peaks):
    """Times `calls` back-to-back T-token layer calls per step (inputs resident), then the same
    steps with an event pair around every launch (per-kernel durations), then end to end through
    the host-buffer entry point (host copies inside every call).  Returns the numbers."""
    hbm_peak, bf16_peak, peak_kind = peaks
    tokens_per_step = calls * T
    xd = torch.from_numpy(xs.view(np.int16)).cuda()
    y = torch.empty((tokens_per_step, D), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        for c in range(calls):
            k3.k3moe_layer_forward(layer, xd[c * T:(c + 1) * T], T, y[c * T:(c + 1) * T], stream)

    for _ in range(args.warmup):
        step()
    k3.k3moe_sync(layer)
    # Decode configurations: the step's layer calls are captured once as a CUDA graph by the
    # library (k3moe_graph_create) and the timed steps replay it (a decode loop's launch overhead
    # leaves the host; the calls and their bytes are the eager calls', which a GPU test checks).
    # The eager steps are timed too.
    graph = None
    if T < 512 and not args.eager:
        graph = k3.k3moe_graph_create(layer, xd, T, calls, y, stream)
        k3.k3moe_graph_launch(graph, stream)
        k3.k3moe_sync(layer)

    def timed(n_steps, use_graph):
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_steps):
            if use_graph:
                k3.k3moe_graph_launch(graph, stream)
            else:
                step()
        e1.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        return e0.elapsed_time(e1)

    ms = timed(args.steps, graph is not None)
    k3.k3moe_sync(layer)  # any device-side wait that gave up would make the timing invalid
    ms_eager = timed(args.steps, False) if graph is not None else ms
    k3.k3moe_sync(layer)
    if graph is not None:
        k3.k3moe_graph_destroy(graph)
    # per-kernel durations: the same steps again with an event pair around every launch (the
    # events sit between kernels and stop programmatic launch overlap, so the headline timing
    # above runs without them)
    k3.k3moe_profile(layer, True)
    ms_profiled = timed(args.steps, False)
    prof = k3.k3moe_profile_read(layer)
    k3.k3moe_profile(layer, False)
    value, ms = job_throughput(tokens_per_step * args.steps, ms, pg)
    value_eager, ms_eager = job_throughput(tokens_per_step * args.steps, ms_eager, pg)

    # distinct experts touched (algorithmic weight bytes): counted from the actual routing
    idx = torch.empty((tokens_per_step, K), dtype=torch.int32, device="cuda")
    w = torch.empty((tokens_per_step, K), dtype=torch.float32, device="cuda")
    for c in range(calls):
        k3.k3moe_router_topk(layer, xd[c * T:(c + 1) * T], T, idx[c * T:(c + 1) * T], w[c * T:(c + 1) * T], stream)
    torch.cuda.synchronize()
    idx_h = idx.cpu().numpy()
    distinct = sum(len(np.unique(idx_h[c * T:(c + 1) * T])) for c in range(calls))
    weight_bytes_per_step = distinct * EXPERT_BYTES
    roofline = _roofline(prof, T, distinct / calls, hbm_peak, bf16_peak, peak_kind)
    launches = sum(v[1] for v in prof.values())

    # end to end through the C ABI with host buffers: every call copies its tokens from pinned
    # host memory, runs the layer and copies y back before it returns
    xh = torch.from_numpy(xs.view(np.int16)).pin_memory()
    yh = torch.empty((tokens_per_step, D), dtype=torch.float32).pin_memory()

    def e2e_step():
        for c in range(calls):
            k3.k3moe_layer_forward_host(layer, xh[c * T:(c + 1) * T], T, yh[c * T:(c + 1) * T], stream)

    e2e_step()
    e2e_steps = max(1, min(args.steps, 3))
    if pg:
        pg.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    e2e_val = job_rate_min(tokens_per_step * e2e_steps / e2e_s, pg)
    ms_step = ms / args.steps
    bf16_sus, _ = _bf16_sustained()
    layer_tflops = 6.0 * F * D * K * tokens_per_step * args.steps / (ms / 1e3) / 1e12
    return {
        "value": round(value, 3), "unit": "tokens/s", "ms_per_step": round(ms_step, 4),
        "calls_per_step": calls, "tokens_per_step": tokens_per_step, "us_per_call": round(1e3 * ms_step / calls, 2),
        "launch": ("one CUDA graph per step: the step's layer calls captured once by k3moe_graph_create, "
                   "then replayed with k3moe_graph_launch" if graph is not None else "eager layer calls"),
        "eager": {"value": round(value_eager, 3), "ms_per_step": round(ms_eager / args.steps, 4)},
        "weight_gbs": round(weight_bytes_per_step * args.steps * (pg.get_world_size() if pg else 1)
                            / (ms / 1e3) / 1e9, 1),
        "weight_pct_of_hbm_peak": round(100 * weight_bytes_per_step * args.steps / (ms / 1e3) / 1e9 / hbm_peak, 1),
        "weight_pct_of_nominal_8tbs": round(100 * weight_bytes_per_step * args.steps / (ms / 1e3) / 1e9
                                            / NOMINAL_HBM_GBS, 1),
        "distinct_experts_per_call": round(distinct / calls, 2),
        # the whole layer's expert flops (6 f d per pick: gate, up, down) over its time, against
        # the measured bf16 peaks (burst, and sustained under the power cap)
        "layer_tflops": round(layer_tflops, 1),
        "layer_pct_of_bf16": {"burst": round(100 * layer_tflops / bf16_peak, 1),
                              "sustained": round(100 * layer_tflops / bf16_sus, 1),
                              "peak_kind": peak_kind},
        "roofline": roofline,
        "kernel_ms_per_launch": {k: round(v[0] / v[1], 5) for k, v in prof.items() if v[1]},
        "kernel_timing": f"event pairs around every launch, second pass of the same {args.steps} steps "
                         f"({round(ms_profiled / args.steps, 4)} ms/step with the events in place)",
        "gpu_launches": int(launches),
        "e2e": {"value": round(e2e_val, 3), "unit": "tokens/s",
                "h2d_bytes_per_step": tokens_per_step * D * 2, "d2h_bytes_per_step": tokens_per_step * D * 4,
                "timing": f"wall clock of {e2e_steps} steps, each {calls} calls of k3moe_layer_forward_host "
                          f"(C ABI, host buffers: H2D of x from pinned memory, the layer, D2H of y, one "
                          f"synchronisation per call)"},
    }


def run_b300(args):
    import torch
    import synth
    import mxfp4_routed_expert_06_b300 as k3

    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    peaks = _peaks()
    # the headline workload first, then (default run) the metric's other two token counts
    names = ["decode1", "decode64", "prefill4096"] if args.workload == "all" else [args.workload]
    clocks = ClockSampler(local)
    clocks.start()
    results = {}
    layer, layer_kind = None, None
    for name in names:
        T = WORKLOADS[name]["T"]
        kind = "prefill" if name == "prefill4096" else "decode"
        if layer_kind != kind:
            if layer is not None:
                k3.k3moe_layer_free(layer)
                torch.cuda.empty_cache()
            bias = synth.hot_bias(SEED, 0, args.experts, 32, 2.0) if kind == "prefill" else None
            layer = build_layer(torch, k3, 4096 if kind == "prefill" else 64, bias, args.experts)
            layer_kind = kind
        if T == 1:
            calls = args.tokens_per_step
        elif T == 64:
            calls = max(1, args.tokens_per_step // 64)
        else:
            calls = 1
        # seeded tokens, distinct per rank and per workload
        xs = synth.tokens_bf16(SEED, 0, rank * 10_000_000 + 1_000_000 * len(results), calls * T, D)
        results[name] = measure(torch, k3, layer, T, calls, xs, args, pg, rank, peaks)
    clk = clocks.stop()
    k3.k3moe_layer_free(layer)

    out = None
    if rank == 0:
        head_name = names[0]
        head = results[head_name]
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            cpu = {n: cpu_baselines(n, args.cpu_seconds) for n in names}
        out = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4 weights -> f16 mma, f32 accumulate",
            "data": "synthetic (seeded splitmix64 experts, N(0,1) bf16 tokens, N(0,1/d) router)",
            "impl": "b300",
            "config": {"workload": WORKLOADS[head_name]["desc"] + _profiling_case(args),
                       "calls_per_step": head["calls_per_step"], "tokens_per_step": head["tokens_per_step"],
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": L2_NOTE[head_name]},
        }
        for key in ("weight_gbs", "weight_pct_of_hbm_peak", "weight_pct_of_nominal_8tbs", "layer_tflops",
                    "layer_pct_of_bf16", "distinct_experts_per_call", "roofline",
                    "kernel_ms_per_launch", "kernel_timing", "gpu_launches", "e2e"):
            out[key] = head[key]
        out["config"]["launch"] = head["launch"]
        out["eager"] = head["eager"]
        out["clocks"] = clk
        out["cpu_baseline"] = None if cpu is None else cpu[head_name]["all_cores"]
        if len(names) > 1:
            out["gpu_launches"] = int(sum(results[n]["gpu_launches"] for n in names))
            out["configs"] = {}
            for n in names:
                r = dict(results[n])
                r["workload"] = WORKLOADS[n]["desc"]
                r["l2"] = L2_NOTE[n]
                r["cpu_baseline"] = None if cpu is None else cpu[n]
                out["configs"][n] = r
        elif cpu is not None:
            out["cpu_baseline_1thread"] = cpu[head_name]["one_thread"]
    if pg:
        pg.destroy_process_group()
    return out


def run_stack4(args):
    """Four stacked layers in cache mode: a step is tokens_per_step T=1 tokens, each through all
    four layers (the caller's residual between them); the budget sets the device cache size."""
    import torch
    import synth
    import mxfp4_routed_expert_06_b300 as k3

    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    n_layers = 4
    budget = int(args.budget_gb * 1e9)
    cache = k3.k3moe_cache_create(budget, EXPERT_BYTES)
    if args.device_lru:
        k3.k3moe_cache_set_device_lru(cache, 1)
    nb, sb = synth.expert_bytes(D, F)
    layers = []
    for l in range(n_layers):
        dn = torch.empty(E * nb, dtype=torch.uint8, device="cuda")
        ds = torch.empty(E * sb, dtype=torch.uint8, device="cuda")
        synth.experts_to_device(SEED, l, 0, E, D, F, dn.data_ptr(), ds.data_ptr())
        Wr = torch.from_numpy(synth.router_weights(SEED, l, E, D)).cuda()
        layers.append(k3.k3moe_pack_experts(k3.dims(D, F, E, K, 1), dn, ds, 1, Wr, None, cache))
        k3.k3moe_set_option(layers[-1], k3.K3MOE_OPT_MISS_PATH,
                            k3.K3MOE_MISS_ZERO_COPY if args.miss_path == "zero-copy" else k3.K3MOE_MISS_COPY_ENGINE)
        del dn, ds, Wr
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    n_tok = args.tokens_per_step
    xs = synth.tokens_bf16(SEED, 0, rank * 10_000_000, n_tok, D)
    xd = torch.from_numpy(xs.view(np.int16)).cuda()
    ys = torch.empty((n_tok, n_layers, D), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    resid = torch.empty((1, D), dtype=torch.int16, device="cuda")
    xin = torch.empty((1, D), dtype=torch.int16, device="cuda")
    idx = torch.empty((1, K), dtype=torch.int32, device="cuda")
    wts = torch.empty((1, K), dtype=torch.float32, device="cuda")

    def record_trace():
        # the expert set each call of a step looks up, from the library's own top-k on the same
        # layer inputs (one untimed step)
        trace = []
        for t in range(n_tok):
            x = xd[t:t + 1]
            resid.copy_(x)
            for l, L in enumerate(layers):
                k3.k3moe_router_topk(L, x, 1, idx, wts, stream)
                trace.append([l * E + int(e) for e in np.unique(idx.cpu().numpy())])
                y = ys[t, l:l + 1]
                k3.k3moe_layer_forward(L, x, 1, y, stream)
                k3.k3moe_residual_rmsnorm(y, resid, 1, D, 1e-6, resid, xin, stream)
                x = xin
        torch.cuda.synchronize()
        return trace

    # Prefetch of the next call's experts while this call computes (k3moe_cache_prefetch):
    # "trace" lists the set the next call will look up (recorded in an untimed step before the
    # warm-up: the most any predictor can gain); "router" guesses it with the next layer's router
    # on this layer's input (for the next token's first layer, on that token: exact).
    trace = record_trace() if args.prefetch == "trace" else None
    pidx = torch.empty((1, K), dtype=torch.int32, device="cuda")
    pidx_host = torch.empty((1, K), dtype=torch.int32).pin_memory()
    guess_ready = torch.cuda.Event()

    def step():
        # layer 0 takes the token; then r = bf16(r + y) and the next layer takes RMSNorm(r)
        c = 0
        for t in range(n_tok):
            x = xd[t:t + 1]
            resid.copy_(x)
            for l, L in enumerate(layers):
                nxt = layers[(l + 1) % n_layers]
                if args.prefetch == "router":
                    guess_in = x if l + 1 < n_layers else xd[(t + 1) % n_tok:(t + 1) % n_tok + 1]
                    k3.k3moe_router_topk(nxt, guess_in, 1, pidx, wts, stream)
                    pidx_host.copy_(pidx, non_blocking=True)
                    guess_ready.record(stream)
                y = ys[t, l:l + 1]
                k3.k3moe_layer_forward(L, x, 1, y, stream)
                # the FFN of this call is still running while the next call's experts come in
                if args.prefetch == "router":
                    guess_ready.synchronize()  # the router and the copy only (the FFN is queued after)
                    k3.k3moe_cache_prefetch(nxt, np.unique(pidx_host.numpy()))
                elif args.prefetch == "trace":
                    nc = (c + 1) % len(trace)
                    k3.k3moe_cache_prefetch(nxt, [e - ((nc % n_layers) * E) for e in trace[nc]])
                k3.k3moe_residual_rmsnorm(y, resid, 1, D, 1e-6, resid, xin, stream)
                x = xin
                c += 1

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    k3.k3moe_cache_reset_stats(cache)
    clocks = ClockSampler(local)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    st = k3.k3moe_cache_stats(cache)
    # per-kernel durations: one more step with event pairs around every launch (the events
    # stop programmatic launch overlap, so the timed steps above run without them)
    for L in layers:
        k3.k3moe_profile(L, True)
    step()
    torch.cuda.synchronize()
    prof = {}
    for L in layers:
        for kname, (kms, kn) in k3.k3moe_profile_read(L).items():
            a = prof.setdefault(kname, [0.0, 0])
            a[0] += kms
            a[1] += kn
        k3.k3moe_profile(L, False)
    # Cache-policy study: the expert set each call of a step looks up (recorded in an untimed
    # pass with the library's own top-k on the same layer inputs), replayed as the warm-up and
    # timed steps through the same number of slots under LRU (the device cache's policy),
    # Belady's MIN and random replacement; hit rates over the timed steps.
    slots = budget // EXPERT_BYTES
    if trace is None:
        trace = record_trace()
    study = {}
    for name, pol in (("lru", k3.K3MOE_POLICY_LRU), ("min", k3.K3MOE_POLICY_MIN), ("random", k3.K3MOE_POLICY_RANDOM)):
        warm = k3.k3moe_cache_simulate(trace * args.warmup, slots, pol, SEED)
        full = k3.k3moe_cache_simulate(trace * (args.warmup + args.steps), slots, pol, SEED)
        h, m = full["hits"] - warm["hits"], full["misses"] - warm["misses"]
        study[name] = {"hits": h, "misses": m, "hit_rate": round(h / max(1, h + m), 4)}
    # without prefetch the device cache must count what the simulated LRU counts
    study["lru_equals_device"] = ((study["lru"]["hits"], study["lru"]["misses"]) == (st["hits"], st["misses"])
                                  if args.prefetch == "none" else None)
    value, ms = job_throughput(n_tok * args.steps, ms, pg)
    hbm_peak, _, peak_kind = _peaks()
    gu_ms, gu_n = prof.get("gateup", (0.0, 0))
    achieved = K * GATEUP_BYTES / (gu_ms / gu_n / 1e3) / 1e9 if gu_n else None
    out = None
    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4 weights -> f16 mma, f32 accumulate",
            "data": "synthetic (seeded splitmix64 experts, N(0,1) bf16 tokens, N(0,1/d) router)",
            "impl": "b300",
            "config": {"workload": WORKLOADS["stack4"]["desc"], "budget_gb": args.budget_gb,
                       "miss_path": "device-side LRU + zero-copy" if args.device_lru else args.miss_path,
                       "prefetch": args.prefetch,
                       "cache_slots": budget // EXPERT_BYTES, "tokens_per_step": n_tok, "layers": n_layers,
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": "inputs larger than L2: 62.9 GB pool"},
            "cache": {"hits": st["hits"], "misses": st["misses"], "evictions": st["evictions"],
                      "prefetched": st["prefetched"],
                      "hit_rate": round(st["hits"] / max(1, st["hits"] + st["misses"]), 4),
                      "h2d_gb": round(st["h2d_bytes"] / 1e9, 3),
                      "h2d_gbs_of_copy_time": round(st["h2d_bytes"] / 1e6 / max(st["h2d_ms"], 1e-9), 2),
                      "h2d_gbs_of_wall": round(st["h2d_bytes"] / 1e6 / ms, 2),
                      "policy_study": study},
            "roofline": {"bound": "hbm", "kernel": "gateup_kernel (gate/up + SwiGLU, register decode)",
                         "achieved": None if achieved is None else round(achieved, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": None if achieved is None else round(achieved / hbm_peak, 4),
                         "peak_kind": f"{peak_kind} (HBM copy peak)", "traffic": None},
            "kernel_ms_per_launch": {k: round(v[0] / v[1], 5) for k, v in prof.items() if v[1]},
            "gpu_launches": int(sum(v[1] for v in prof.values())),
            "clocks": clk,
            "cpu_baseline": None,
        }
    for L in layers:
        k3.k3moe_layer_free(L)
    k3.k3moe_cache_destroy(cache)
    if pg:
        pg.destroy_process_group()
    return out


# ---------------------------------------------------------------------- oracle arm ---

def _oracle_tokens(n_tokens, rank_offset=0):
    """The oracle on n_tokens single-token calls of the K3 layer: returns seconds and threads used."""
    import oracle
    import synth
    Wr = synth.router_weights(SEED, 0, E, D)
    xs = synth.tokens_bf16(SEED, 0, rank_offset, n_tokens, D)
    # expert bytes are regenerated on the host; that is input preparation, not timed
    t_total = 0.0
    for t in range(n_tokens):
        t0 = time.perf_counter()
        idx, w, _, _ = oracle.router(xs[t:t + 1], Wr, None, K)
        oracle.bucket(idx, E)
        t_total += time.perf_counter() - t0
        nibs, scls = _expert_blocks(idx[0])
        t0 = time.perf_counter()
        oracle.moe(xs[t:t + 1], w, nibs, scls, F)
        t_total += time.perf_counter() - t0
    return t_total, oracle.max_threads()


def _expert_blocks(ids, seed=SEED):
    import synth
    nibs, scls = [], []
    for e in ids.tolist():
        n, s = synth.experts(seed, 0, e, e + 1, D, F)
        nibs.append(n[0])
        scls.append(s[0])
    return nibs, scls


def _oracle_batch(router_tokens, y_seconds, bias=None):
    """The oracle on one multi-token call, sampled: router + top-k and bucketing on router_tokens
    tokens (timed once), then the expert FFNs and combine token by token until y_seconds of FFN
    time have passed (at least one token).  Tokens are independent, so seconds per token =
    router part / router_tokens + FFN part / FFN tokens.  Returns (seconds per token, threads,
    FFN tokens)."""
    import oracle
    import synth
    Wr = synth.router_weights(SEED, 0, E, D)
    xs = synth.tokens_bf16(SEED, 0, 5_000_000, router_tokens, D)
    t0 = time.perf_counter()
    idx, w, _, _ = oracle.router(xs, Wr, bias, K)
    oracle.bucket(idx, E)
    t_router = time.perf_counter() - t0
    t_ffn, n_y = 0.0, 0
    while n_y < router_tokens and (n_y == 0 or t_ffn < y_seconds):
        nibs, scls = _expert_blocks(idx[n_y])
        t0 = time.perf_counter()
        oracle.moe(xs[n_y:n_y + 1], w[n_y:n_y + 1], nibs, scls, F)
        t_ffn += time.perf_counter() - t0
        n_y += 1
    return t_router / router_tokens + t_ffn / n_y, oracle.max_threads(), n_y


def _one_cpu_baseline(name, threads, seconds):
    import oracle
    oracle.build()
    oracle.set_threads(threads)
    try:
        if name == "decode1":
            n = 1
            sec, cores = _oracle_tokens(n)
            if sec < seconds * 0.5:
                n = max(1, min(64, int(n * seconds * 0.5 / max(sec, 1e-3))))
                sec, cores = _oracle_tokens(n, 100)
            return {"value": round(n / sec, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                    "sample": f"{n} single-token K3 layer calls (router over 896 experts, top-16, bucketing and "
                              f"16 expert FFNs each), fp64 scalar MXFP4 decode, {sec:.1f} s"}
        T = WORKLOADS[name]["T"]
        bias = synth_bias() if name == "prefill4096" else None
        r_tok = T if threads > 1 else min(T, 64)
        per_tok, cores, n_y = _oracle_batch(r_tok, seconds * 0.5, bias)
        return {"value": round(1.0 / per_tok, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": f"one {T}-token call sampled: router, top-16 and bucketing on {r_tok} tokens, the "
                          f"16 expert FFNs and combine on {n_y} of them; seconds per token = router part / "
                          f"{r_tok} + FFN part / {n_y} (tokens are independent, so the whole call "
                          f"extrapolates linearly); fp64 scalar MXFP4 decode"}
    finally:
        oracle.set_threads(os.cpu_count() or 1)


def synth_bias():
    import synth
    return synth.hot_bias(SEED, 0, E, 32, 2.0)


def cpu_baselines(name, seconds):
    """The oracle as it stands, on bounded samples of the workload: all host cores, then 1 thread."""
    return {"all_cores": _one_cpu_baseline(name, os.cpu_count() or 1, seconds),
            "one_thread": _one_cpu_baseline(name, 1, seconds / 2)}


def run_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    per_step = 1
    for _ in range(args.warmup):
        _oracle_tokens(per_step, 500)
    total = 0.0
    cores = 1
    for s in range(args.steps):
        sec, cores = _oracle_tokens(per_step, 1000 + s)
        total += sec
    value = per_step * args.steps / total
    wl = WORKLOADS["decode1"]
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (same generator as the b300 arm)",
        "impl": "reference",
        "config": {"workload": wl["desc"], "calls_per_step": per_step, "tokens_per_step": per_step,
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} single-token layer call per step (bounded sample of the "
                                   f"1000-token decode workload)"},
        "e2e": {"value": round(value, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(WORKLOADS),
                    help="all (default): the single-token decode headline, then T=64 and T=4096 under 'configs'")
    ap.add_argument("--tokens-per-step", type=int, default=None,
                    help="tokens per step of the decode workloads: T=1 calls (default 1000; 256 for stack4); "
                         "the T=64 workload runs this many tokens in T=64 calls")
    ap.add_argument("--budget-gb", type=float, default=8.0, help="stack4: device cache budget (1 GB = 1e9 B)")
    ap.add_argument("--miss-path", default="copy-engine", choices=["copy-engine", "zero-copy"],
                    help="stack4: how missed experts reach their slots (K3MOE_OPT_MISS_PATH)")
    ap.add_argument("--device-lru", action="store_true",
                    help="stack4: the cache keeps its LRU state on the device (k3moe_cache_set_device_lru)")
    ap.add_argument("--prefetch", choices=["none", "trace", "router"], default="none",
                    help="stack4: while a call computes, prefetch the next call's experts (k3moe_cache_prefetch): "
                         "'trace' = the set it will look up (recorded before the warm-up), 'router' = the next "
                         "layer's router on this layer's input")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="decode configurations: time eager layer calls only (default: the step's calls "
                         "replayed as one captured CUDA graph, eager timed beside it)")
    ap.add_argument("--experts", type=int, default=E,
                    help="experts resident (default 896); fewer gives a small case with the same per-call work "
                         "at T=1, for profiler captures")
    ap.add_argument("--f", type=int, default=F,
                    help="expert intermediate width (default 1536, a multiple of 128); a narrow FFN gives a "
                         "small case in which the router still does the full layer's work, for profiler captures")
    args = ap.parse_args()
    if args.f != F:
        _set_ffn_width(args.f)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.prefetch != "none" and args.device_lru:
        ap.error("--prefetch needs the host-side LRU bookkeeping (not --device-lru)")
    if args.tokens_per_step is None:
        args.tokens_per_step = 256 if args.workload == "stack4" else 1000
    if args.impl == "reference":
        out = run_reference(args)
    elif args.workload == "stack4":
        out = run_stack4(args)
    else:
        out = run_b300(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
