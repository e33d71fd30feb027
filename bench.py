"""Benchmark of the fused MoE forward (route + align + permute + SwiGLU
grouped GEMM + down-projection grouped GEMM + top-k weight-and-reduce).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixtral_prefill]

One step = one pass of the whole path over one batch of synthetic inputs of
the named workload (default: the Mixtral-8x7B-shape layer, prefill M=4096).
Weights and inputs are resident in HBM before timing; the weights (2.8 GB)
exceed the 129 MB L2, so no flush is needed between steps.

With the default workload the line also carries, under "configs", every
other workload of the layer family measured the same way (its own step
count, stated): the tiny layer (warm, and cold-L2 with a 256 MB write
between steps), the Mixtral-shape M=16 decode, DeepSeek-V3-shape M=64 and
M=8192, the Qwen-MoE shape with skewed routing (Zipf popularity and the
literal Zipf draw), and the batched layout -- each with its step roofline
fraction, its dominant kernel's roofline and a bounded-sample CPU oracle
baseline.  Roofline peaks: the measured burst bf16 GEMM rate and the
measured copy bandwidth (every kernel here is timed in a region well under
a second); the sustained and the nominal dense peaks are given beside them.

--impl reference times the CPU oracle (test infrastructure, fp64 numpy) on a
bounded sample of the same workload on the host cores.

Multi-GPU: every rank runs an independent replica on its own batch (the
path shards by tokens with no collective); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_ffn_softmax_gb300 import workloads as wl  # noqa: E402

METRIC = "fused-MoE fwd tokens/s and TFLOP/s (1×GB300), % of roofline"


NOMINAL_DENSE_BF16_TFLOPS = 2250.0   # GB300 datasheet, dense bf16 (context only)
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def measured_traffic(kernel, workload):
    """(DRAM bytes per launch, note) from the committed record
    profiles/traffic_<kernel>_<workload>.json (written from an ncu export by
    mixture_experts_ffn_softmax_gb300/ncu_traffic.py).  The bytes are None
    when there is no record or when the kernel source has changed since the
    counters were taken (the record holds the source's hash)."""
    import hashlib
    rec_path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.json")
    if not os.path.exists(rec_path):
        return None, "no ncu record"
    try:
        with open(rec_path) as f:
            rec = json.load(f)
        src = os.path.join(ROOT, rec["source"])
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        if rec["kernel"] != kernel or rec["workload"] != workload:
            return None, "record names another kernel or workload"
        if sha != rec["source_sha256_16"]:
            return None, f"stale: {rec['source']} changed since the ncu capture"
        return int(rec["traffic_bytes_per_launch"]), (
            f"profiles/traffic_{kernel}_{workload}.json, {rec['source']} "
            f"sha256[:16] {rec['source_sha256_16']}")
    except (OSError, KeyError, ValueError) as e:
        return None, f"unreadable record: {e}"


# ----------------------------------------------------------- distributed --
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_rate(units_per_rank, world, ms_max):
    """Whole-job throughput: every rank processes units_per_rank per step and
    the job's step lasts as long as its slowest rank (ms_max, already the
    maximum over ranks)."""
    return units_per_rank * world / (ms_max / 1e3)


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads --
def algorithmic(spec, ids_np):
    """FLOPs = 6 R H I; bytes = touched expert weights + x + out + logits."""
    touched = int(np.unique(ids_np).size)
    wbytes = touched * 3 * spec.H * spec.I * 2
    if spec.bias:
        wbytes += touched * (2 * spec.I + spec.H) * 2
    io = spec.M * spec.H * 2 * 2 + spec.M * spec.E * 4
    return spec.flops(), wbytes + io, touched


def kernel_work(name, H, I, E, k, M, R, touched, bias=False):
    """Algorithmic (FLOPs, bytes) of one launch of a kernel of the step.
    R routed rows (M*k, or the valid rows of the batched layout), `touched`
    experts with at least one row; bf16 weights and activations, fp32 item
    rows.  GEMM1: 4HI FLOPs per row; its touched experts' w13 (4HI bytes each)
    + the rows read (2H) + z written (2I).  GEMM2: 2HI FLOPs per row; w2
    (2HI bytes each) + z read (2I) + the fp32 (4H) or bf16 (2H) row written.
    Gather 2H read per token (each token row once) + 2H written per row (the
    batched layout passes M = R); reduce 4kH read + 2H written per
    token; route 4E read + 8k written per token; align 4 B read twice and
    8 B written per row.  The small-call kernels: GEMM1 as above + the fp32
    token accumulator zeroed (4H per token); GEMM2 its w2, z read, and per
    token the accumulator read (4H) and y written (2H).  Returns None for a
    kernel not listed."""
    b13 = touched * 2 * I * 2 if bias else 0
    b2 = touched * H * 2 if bias else 0
    if name == "gemm1_swiglu":
        return 4.0 * R * H * I, touched * 4 * H * I + b13 + R * (2 * H + 2 * I)
    if name == "gemm2_sorted":
        return 2.0 * R * H * I, touched * 2 * H * I + b2 + R * (2 * I + 4 * H)
    if name == "gemm2_atomic":
        return 2.0 * R * H * I, touched * 2 * H * I + b2 + R * 2 * I + M * H * 4
    if name == "gemm2_rows_bf16":
        return 2.0 * R * H * I, touched * 2 * H * I + b2 + R * (2 * I + 2 * H)
    if name == "small_gemm1":
        return 4.0 * R * H * I, touched * 4 * H * I + b13 + R * (2 * H + 2 * I) + M * 4 * H
    if name == "small_gemm2":
        return 2.0 * R * H * I, touched * 2 * H * I + b2 + R * 2 * I + M * 6 * H
    if name == "gather_rows":
        return 0.0, (M + R) * 2 * H
    if name == "reduce_sorted":
        return 0.0, M * (4 * k * H + 2 * H)
    if name == "cast_f32_bf16":
        return 0.0, M * 6 * H
    if name == "route":
        return 0.0, M * (4 * E + 8 * k)
    if name.startswith("align") or name == "batched_plan":
        return 0.0, R * 16
    return None


def roofline_of(flops, nbytes, seconds, pk):
    """Roofline of work (flops, bytes) done in `seconds`: t_roof = max(flops /
    burst bf16 peak, bytes / copy bandwidth); frac = t_roof / seconds."""
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_tc >= t_hbm:
        ach = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(t_tc / seconds, 4),
                "frac_of_sustained_peak": round(ach / pk["bf16_tflops_sustained"], 4),
                "frac_of_nominal_dense_peak": round(ach / NOMINAL_DENSE_BF16_TFLOPS, 4)}
    ach = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(t_hbm / seconds, 4)}


def dominant_kernel(kern, work):
    """The kernel with the largest share of the step's device time, with its
    roofline.  kern: name -> {"launches", "avg_us"} over the profiled steps;
    work: name -> (flops, bytes) per launch."""
    total = sum(v["launches"] * v["avg_us"] for v in kern.values())
    name = max(kern, key=lambda n: kern[n]["launches"] * kern[n]["avg_us"])
    v = kern[name]
    return name, v["launches"] * v["avg_us"] / max(total, 1e-9), work.get(name)


def time_steps_cold(step, K, W, flush):
    """Per-step device time with L2 flushed before every step: a write of
    `flush` (larger than L2) between steps, outside the timed events.
    Returns the summed milliseconds of the K timed steps."""
    for _ in range(W):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(K):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        step()
        e1.record(s)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


class OurStep:
    reduce = "auto"

    def __init__(self, spec, device, weights_from=None):
        """weights_from: the input dict of another workload of the same layer
        (same E, H, I, seed): its weights are used instead of drawing them
        again (they are the same draws)."""
        import mixture_experts_ffn_softmax_gb300 as pkg
        self.pkg = pkg
        self.spec = spec
        self.d = wl.make_moe_inputs(spec, device=device, weights=weights_from is None)
        if weights_from is not None:
            for key in ("w13", "w2", "w13_bias", "w2_bias"):
                self.d[key] = weights_from[key]
        M, E, k = spec.M, spec.E, spec.top_k
        self.w = torch.empty(M, k, dtype=torch.float32, device=device)
        self.ids = torch.empty(M, k, dtype=torch.int32, device=device)
        self.ws = pkg.alloc_workspace(pkg.workspace_size(M, spec.H, spec.I, E, k), device)
        self.out = torch.empty_like(self.d["hidden"])

    def __call__(self, hidden=None, logits=None):
        s, d, pkg = self.spec, self.d, self.pkg
        pkg.moe_route(d["router_logits"] if logits is None else logits, s.top_k,
                      s.routing_method, s.renormalize, s.k_group, s.group_count,
                      s.group_select_mode, s.routed_scaling_factor, self.w, self.ids)
        pkg.moe_forward(d["hidden"] if hidden is None else hidden, self.w, self.ids, d["w13"],
                        d["w2"], d["w13_bias"], d["w2_bias"], self.ws, self.out,
                        reduce=self.reduce)
        return self.out


def _graph_ms(step, K, W, world):
    """The same step captured once into a CUDA graph and replayed (launch
    overhead removed; matters for the small shapes)."""
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        step()
    torch.cuda.current_stream().wait_stream(gs)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    ms = max_over_ranks(time_steps(graph.replay, K, W, world) / K, world)
    del graph
    return ms


def _steps_for(step, K, W, world, target_ms=50.0):
    """At least K timed steps, more for short steps (about target_ms of timed
    work, at most 1000 steps), from a 3-step probe after the warm-up."""
    probe = time_steps(step, 3, W, world) / 3
    return int(min(1000, max(K, round(target_ms / max(probe, 1e-3)))))


def _profile(step, n):
    import mixture_experts_ffn_softmax_gb300 as pkg
    pkg.profiler_start()
    for _ in range(n):
        step()
    prof = pkg.profiler_stop()
    return {k: {"launches": v[0] // n, "avg_us": 1e3 * v[1] / max(v[0], 1)}
            for k, v in prof.items()}


def _summary(kern, work, ms, flops, nbytes, pk):
    """Step roofline + dominant kernel roofline of one measured config."""
    step_roof = roofline_of(flops, nbytes, ms * 1e-3, pk)
    t_roof = max(flops / (pk["bf16_tflops"] * 1e12), nbytes / (pk["hbm_gbs"] * 1e9)) * 1e3
    name, share, w = dominant_kernel(kern, work)
    dom = {"kernel": name, "avg_us": round(kern[name]["avg_us"], 2),
           "share_of_step": round(share, 4)}
    if w is not None:
        dom.update(roofline_of(w[0], w[1], kern[name]["avg_us"] * 1e-6, pk))
        dom["algorithmic_flops"], dom["algorithmic_bytes"] = w[0], int(w[1])
    return {"t_roof_ms": round(t_roof, 4), "frac": step_roof["frac"],
            "bound": step_roof["bound"]}, dom


def measure_config(spec, device, K, W, world, pk, weights_from=None, cold_l2=False,
                   cpu=True, cpu_budget=3.0, graph=True):
    """One contiguous-layout workload measured like the headline: timed steps
    (device-resident inputs), per-kernel events, the step roofline, the
    dominant kernel's roofline, a CUDA-graph replay, optionally a cold-L2
    timing, and a bounded-sample CPU oracle baseline."""
    import mixture_experts_ffn_softmax_gb300 as pkg
    step = OurStep(spec, device, weights_from=weights_from)
    Kc = _steps_for(step, K, W, world)
    n0 = pkg.launch_count()
    ms = max_over_ranks(time_steps(step, Kc, W, world) / Kc, world)
    launches = (pkg.launch_count() - n0) // (Kc + W)
    flops, nbytes, touched = algorithmic(spec, step.ids.cpu().numpy())
    kern = _profile(step, min(Kc, 50))
    work = {n: kernel_work(n, spec.H, spec.I, spec.E, spec.top_k, spec.M, spec.R, touched,
                           spec.bias) for n in kern}
    work = {n: w for n, w in work.items() if w is not None}
    roof_step, dom = _summary(kern, work, ms, flops, nbytes, pk)
    out = {"workload": spec.name, "M": spec.M, "H": spec.H, "I": spec.I, "E": spec.E,
           "top_k": spec.top_k, "routing": spec.routing_method, "steps": Kc,
           "ms_per_step": round(ms, 4), "tokens_per_s": round(job_rate(spec.M, world, ms), 1),
           "tflops": round(flops * world / (ms / 1e3) / 1e12, 2), "experts_touched": touched,
           "algorithmic_bytes": int(nbytes), "roofline_step": roof_step,
           "dominant_kernel": dom, "gpu_launches": launches,
           "kernels_us": {k: round(v["avg_us"], 2) for k, v in kern.items()}}
    if graph:
        gms = _graph_ms(step, Kc, W, world)
        out["graph"] = {"ms_per_step": round(gms, 4),
                        "tokens_per_s": round(job_rate(spec.M, world, gms), 1)}
    if cold_l2:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        cms = max_over_ranks(time_steps_cold(step, Kc, W, flush) / Kc, world)
        out["cold_l2"] = {"ms_per_step": round(cms, 4),
                          "tokens_per_s": round(job_rate(spec.M, world, cms), 1),
                          "roofline_frac": round(roof_step["t_roof_ms"] / cms, 4),
                          "flush": f"{L2_FLUSH_BYTES >> 20} MB written between steps, "
                                   "outside the timed events"}
        del flush
    if cpu and world == 1:
        out["cpu_baseline"] = cpu_baseline(spec, step.d, budget_s=cpu_budget)
    return out, step


class BatchedStep:
    """One pass of the batched-layout forward: (E, T, H) rows with
    expert_num_tokens, per-row weights, invalid rows NaN."""

    def __init__(self, spec, device):
        import mixture_experts_ffn_softmax_gb300 as pkg
        self.pkg = pkg
        self.spec = spec
        self.d = wl.make_batched_inputs(spec, device=device)
        self.ws = pkg.alloc_workspace(pkg.batched_workspace_size(spec.E, spec.T, spec.H, spec.I),
                                      device)
        self.out = torch.empty_like(self.d["x"])
        self.rows = int(self.d["expert_num_tokens"].sum().item())

    def __call__(self, x=None):
        d = self.d
        return self.pkg.moe_forward_batched(d["x"] if x is None else x, d["expert_num_tokens"],
                                            d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                                            d["row_weight"], self.ws, self.out)


def measure_batched(spec, device, K, W, world, pk, cpu=True, cpu_budget=3.0):
    """The batched layout measured like measure_config; FLOPs = 6 * valid
    rows * H * I, bytes = touched experts' weights + valid rows in and out."""
    import mixture_experts_ffn_softmax_gb300 as pkg
    step = BatchedStep(spec, device)
    Kc = _steps_for(step, K, W, world)
    n0 = pkg.launch_count()
    ms = max_over_ranks(time_steps(step, Kc, W, world) / Kc, world)
    launches = (pkg.launch_count() - n0) // (Kc + W)
    R = step.rows
    flops = 6.0 * R * spec.H * spec.I
    touched = int((step.d["expert_num_tokens"] > 0).sum().item())
    nbytes = touched * 3 * spec.H * spec.I * 2 + 2 * R * spec.H * 2
    kern = _profile(step, min(Kc, 50))
    work = {n: kernel_work(n, spec.H, spec.I, spec.E, 1, R, R, touched, spec.bias)
            for n in kern}
    work = {n: w for n, w in work.items() if w is not None}
    roof_step, dom = _summary(kern, work, ms, flops, nbytes, pk)
    gms = _graph_ms(step, Kc, W, world)
    out = {"workload": spec.name, "E": spec.E, "T": spec.T, "H": spec.H, "I": spec.I,
           "valid_rows": R, "steps": Kc, "ms_per_step": round(ms, 4),
           "tokens_per_s": round(job_rate(R, world, ms), 1),
           "tflops": round(flops * world / (ms / 1e3) / 1e12, 2), "experts_touched": touched,
           "algorithmic_bytes": int(nbytes), "roofline_step": roof_step,
           "dominant_kernel": dom, "gpu_launches": launches,
           "kernels_us": {k: round(v["avg_us"], 2) for k, v in kern.items()},
           "graph": {"ms_per_step": round(gms, 4),
                     "tokens_per_s": round(job_rate(R, world, gms), 1)}}
    if cpu and world == 1:
        out["cpu_baseline"] = cpu_baseline_batched(spec, step.d, budget_s=cpu_budget)
    return out, step


def run_batched(args, world, rank, local):
    pk = peaks()
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    spec = wl.BATCHED_SPECS[args.workload]
    K, W = args.steps, args.warmup
    step = BatchedStep(spec, device)
    import mixture_experts_ffn_softmax_gb300 as pkg
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    n0 = pkg.launch_count()
    ms = time_steps(step, K, W, world)
    launches = (pkg.launch_count() - n0) * K // (K + W)
    ck = clocks.stop()
    ms_step = max_over_ranks(ms / K, world)
    R = step.rows
    del step
    m, step = measure_batched(spec, device, K, W, world, pk, cpu=False)
    dom = m["dominant_kernel"]
    roof = {k: dom[k] for k in ("bound", "achieved", "peak", "unit", "frac") if k in dom}
    roof.update({"kernel": dom["kernel"], "traffic": None,
                 "traffic_note": "no ncu record for this kernel and workload",
                 "peak_source": pk["source"] + (" burst bf16" if dom.get("bound") == "tensor"
                                                else " copy")})

    hx = step.d["x"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    dx = torch.empty_like(step.d["x"])

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        y = step(dx)
        hy.copy_(y, non_blocking=True)

    ms_e2e = max_over_ranks(time_steps(e2e_step, K, W, world) / K, world)
    flops = 6.0 * R * spec.H * spec.I
    line = {
        "metric": METRIC, "value": round(job_rate(R, world, ms_step), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{spec.name}: batched layout (E, max_tokens, H)", "E": spec.E,
                   "T": spec.T, "H": spec.H, "I": spec.I, "valid_rows": R,
                   "parallelism": f"replicas x{world}", "l2": "inputs larger than L2"},
        "tflops": round(flops * world / (ms_step / 1e3) / 1e12, 2),
        "roofline_step": m["roofline_step"], "roofline": roof,
        "kernels_us": m["kernels_us"], "graph": m["graph"],
        "gpu_launches": launches, "clocks": ck,
        "e2e": {"value": round(R * world / (ms_e2e / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hy.numel() * 2},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_steps(step, K, W, world, ev_stream=None):
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(K):
        step()
    e1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def workload_config(spec):
    """The workload fields of the line's config, the same on both arms."""
    return {"workload": f"{spec.name}: Mixtral-8x7B-shape MoE layer" if "mixtral" in spec.name
            else spec.name, "M": spec.M, "H": spec.H, "I": spec.I, "E": spec.E,
            "top_k": spec.top_k, "routing": spec.routing_method,
            "renormalize": spec.renormalize}


def run_ours(args, world, rank, local):
    import mixture_experts_ffn_softmax_gb300 as pkg
    pk = peaks()
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    spec = {**wl.SPECS, **wl.PROFILE_SPECS}[args.workload]
    step = OurStep(spec, device)
    K, W = args.steps, args.warmup

    # headline: device-resident inputs
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)                       # sampler up before the timed region
    n0 = pkg.launch_count()
    ms = time_steps(step, K, W, world)
    launches_total = pkg.launch_count() - n0
    ck = clocks.stop()
    launches = launches_total * K // (K + W)   # launches inside the timed region
    ms_step = max_over_ranks(ms / K, world)
    ids_np = step.ids.cpu().numpy()
    flops, nbytes, touched = algorithmic(spec, ids_np)
    tok_s = job_rate(spec.M, world, ms_step)
    tflops = flops * world / (ms_step / 1e3) / 1e12

    # per-kernel timing with events on the launching stream (second timed pass)
    kern = _profile(step, K)
    work = {n: kernel_work(n, spec.H, spec.I, spec.E, spec.top_k, spec.M, spec.R, touched,
                           spec.bias) for n in kern}
    work = {n: w for n, w in work.items() if w is not None}
    roof_step, dom = _summary(kern, work, ms_step, flops, nbytes, pk)
    # The roofline object is GEMM1's (the step's dominant kernel on the
    # prefill shapes; small calls run the small-call GEMM1): algorithmic work
    # per launch / its average event time.
    k1 = "gemm1_swiglu" if "gemm1_swiglu" in kern else "small_gemm1"
    g1 = kern[k1]["avg_us"]
    f1, b1 = work[k1]
    roof = {"kernel": k1, **roofline_of(f1, b1, g1 * 1e-6, pk),
            "algorithmic_flops": f1, "algorithmic_bytes": int(b1),
            "share_of_step": round(kern[k1]["launches"] * g1 / (ms_step * 1e3), 4)}
    traffic, note = measured_traffic(k1, spec.name)
    roof["traffic"] = traffic
    roof["traffic_note"] = note
    roof["peak_source"] = pk["source"] + (
        " burst bf16 (the kernel is timed in a region well under a second)"
        if roof["bound"] == "tensor" else " copy")

    ms_graph = _graph_ms(step, K, W, world)

    # end to end through the C ABI with host buffers (moe_forward_host: the
    # copies of hidden and logits in, routing, the forward, the copy of out
    # back, all inside the call)
    hx = step.d["hidden"].cpu().pin_memory()
    hl = step.d["router_logits"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    st = pkg.HostStaging(spec.M, spec.H, spec.I, spec.E, spec.top_k, device, step.reduce)
    dd = step.d

    def e2e_step():
        pkg.moe_forward_host(hx, hl, dd["w13"], dd["w2"], spec.top_k, spec.routing_method,
                             spec.renormalize, spec.k_group, spec.group_count,
                             spec.group_select_mode, spec.routed_scaling_factor,
                             dd["w13_bias"], dd["w2_bias"], out=hy, staging=st,
                             reduce=step.reduce, stream=torch.cuda.current_stream())

    ms_e2e = max_over_ranks(time_steps(e2e_step, K, W, world) / K, world)
    e2e = {"value": round(spec.M * world / (ms_e2e / 1e3), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": hx.numel() * 2 + hl.numel() * 4,
           "d2h_bytes_per_step": hy.numel() * 2, "ms_per_step": round(ms_e2e, 4),
           "call": "moe_forward_host"}
    del st, hx, hl, hy

    big = spec.M * spec.H * spec.top_k * 2 + 3 * spec.E * spec.H * spec.I * 2 > (129 << 20)
    line = {
        "metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**workload_config(spec), "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (weights of every touched expert are read "
                         "each step)" if big else "inputs fit in L2 (warm)"},
        "tflops": round(tflops, 2),
        "roofline_step": {**roof_step,
                          "peaks": "measured burst bf16 GEMM, measured copy GB/s"},
        "roofline": roof,
        "dominant_kernel": dom,
        "kernels_us": {k: round(v["avg_us"], 2) for k, v in kern.items()},
        "graph": {"ms_per_step": round(ms_graph, 4),
                  "tokens_per_s": round(spec.M * world / (ms_graph / 1e3), 1)},
        "gpu_launches": launches,
        "clocks": ck,
        "e2e": e2e,
    }

    if args.workload == "mixtral_prefill" and not args.no_next_rows:
        line["next_rows"] = measure_next_rows(step, spec, K, W, world, pk)
        line["next_rows"]["weight_only_quantised"] = measure_wq(step, spec, K, W, world, pk)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, step.d, budget_s=args.cpu_budget)

    if args.workload == "mixtral_prefill":
        line["configs"] = measure_all_configs(args, step, device, K, W, world, pk)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_all_configs(args, head_step, device, K, W, world, pk):
    """Every other workload of the layer family, one after the other (each
    freed before the next), measured by measure_config / measure_batched."""
    cpu = world == 1 and not args.no_cpu_baseline
    out = {}

    def free():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    if not args.no_decode:
        out["mixtral_decode"], _ = measure_config(wl.SPECS["mixtral_decode"], device, K, W,
                                                  world, pk, weights_from=head_step.d, cpu=cpu)
    if args.no_configs:
        return out
    out["tiny"], _ = measure_config(wl.SPECS["tiny"], device, K, W, world, pk, cold_l2=True,
                                    cpu=cpu)
    free()
    ds64, st = measure_config(wl.SPECS["deepseek_m64"], device, K, W, world, pk, cpu=cpu)
    out["deepseek_m64"] = ds64
    out["deepseek_m8192"], _ = measure_config(wl.SPECS["deepseek_m8192"], device, K, W, world,
                                              pk, weights_from=st.d, cpu=cpu, graph=False)
    del st
    free()
    q, st = measure_config(wl.SPECS["qwen_skew"], device, K, W, world, pk, cpu=cpu)
    out["qwen_skew"] = q
    out["qwen_skew_lit"], _ = measure_config(wl.SPECS["qwen_skew_lit"], device, K, W, world,
                                             pk, weights_from=st.d, cpu=cpu)
    del st
    free()
    out["batched"], _ = measure_batched(wl.BATCHED_SPECS["batched"], device, K, W, world, pk,
                                        cpu=cpu)
    free()
    return out


def measure_next_rows(step, spec, K, W, world, pk):
    """The rows next to the hot path on the same layer: the router logits GEMM
    (s = x W_g + b_g, W_g ~ N(0, 0.02)), the whole layer from the hidden
    states, the router weight applied to the second layer's input, and one
    expert-parallel holder of half the experts (expert_map)."""
    import mixture_experts_ffn_softmax_gb300 as pkg
    d = step.d
    dev = d["hidden"].device
    g = torch.Generator(device=dev).manual_seed(11)
    wg = (torch.randn(spec.H, spec.E, generator=g, device=dev) * 0.02).bfloat16()
    bg = (torch.randn(spec.E, generator=g, device=dev) * 0.02).bfloat16()
    logits = torch.empty(spec.M, spec.E, device=dev)
    out = {}

    def router():
        pkg.moe_router_logits(d["hidden"], wg, bg, logits)

    ms = max_over_ranks(time_steps(router, K, W, world) / K, world)
    rbytes = spec.M * spec.H * 2 + spec.H * spec.E * 2 + spec.M * spec.E * 4
    out["router_logits"] = {"us": round(ms * 1e3, 2), "hbm_gbs": round(rbytes / (ms * 1e-3) / 1e9, 1),
                            "hbm_frac": round(rbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}

    def layer():
        pkg.moe_router_logits(d["hidden"], wg, bg, logits)
        step(logits=logits)

    ms = max_over_ranks(time_steps(layer, K, W, world) / K, world)
    out["layer_from_hidden"] = {"ms_per_step": round(ms, 4),
                                "tokens_per_s": round(spec.M * world / (ms / 1e3), 1)}

    def on_input():
        pkg.moe_forward(d["hidden"], step.w, step.ids, d["w13"], d["w2"], d["w13_bias"],
                        d["w2_bias"], step.ws, step.out, apply_router_weight_on_input=True)

    ms = max_over_ranks(time_steps(on_input, K, W, world) / K, world)
    out["router_weight_on_input"] = {"ms_per_step": round(ms, 4),
                                     "tokens_per_s": round(spec.M * world / (ms / 1e3), 1)}

    mine = torch.arange(0, spec.E, 2, device=dev)
    emap = torch.full((spec.E,), -1, dtype=torch.int32, device=dev)
    emap[mine] = torch.arange(mine.numel(), dtype=torch.int32, device=dev)
    lw13, lw2 = d["w13"][mine].contiguous(), d["w2"][mine].contiguous()

    def ep_half():
        pkg.moe_forward(d["hidden"], step.w, step.ids, lw13, lw2, None, None, step.ws, step.out,
                        expert_map=emap)

    ms = max_over_ranks(time_steps(ep_half, K, W, world) / K, world)
    local_items = int(torch.isin(step.ids, mine.to(torch.int32)).sum().item())
    fl = 6.0 * local_items * spec.H * spec.I
    out["expert_parallel_half"] = {"ms_per_step": round(ms, 4), "local_items": local_items,
                                   "tflops": round(fl / (ms / 1e3) / 1e12, 2)}
    del lw13, lw2

    # FP8 W8A8: E4M3 weights with per-output-channel scales, activations
    # quantised per row on the GPU; the fp8 tensor peak is the measured
    # burst bf16 peak x 2 (nominal dense fp8 : bf16 = 4.5 : 2.25)
    q = wl.make_fp8_weights(spec, device=dev, per_channel=True)
    ws8 = pkg.alloc_workspace(pkg.workspace_size_fp8(spec.M, spec.H, spec.I, spec.E,
                                                     spec.top_k), dev)

    def fp8():
        pkg.moe_forward_fp8(d["hidden"], step.w, step.ids, q["w13_q"], q["w2_q"],
                            q["w13_scale"], q["w2_scale"], None, None, ws8, step.out)

    ms = max_over_ranks(time_steps(fp8, K, W, world) / K, world)
    pkg.profiler_start()
    for _ in range(K):
        fp8()
    prof = pkg.profiler_stop()
    us = {k: 1e3 * v[1] / max(v[0], 1) for k, v in prof.items()}
    f1 = 4.0 * spec.R * spec.H * spec.I
    peak8 = 2.0 * pk["bf16_tflops"]
    ach = f1 / (us["gemm1_swiglu_fp8"] * 1e-6) / 1e12
    out["fp8_w8a8"] = {"ms_per_step": round(ms, 4),
                       "tokens_per_s": round(spec.M * world / (ms / 1e3), 1),
                       "tflops": round(spec.flops() / (ms / 1e3) / 1e12, 1),
                       "kernels_us": {k: round(v, 2) for k, v in us.items()},
                       "roofline": {"kernel": "gemm1_swiglu_fp8", "bound": "tensor",
                                    "achieved": round(ach, 1), "peak": round(peak8, 1),
                                    "unit": "TFLOP/s", "frac": round(ach / peak8, 4),
                                    "peak_source": "measured burst bf16 x 2 (nominal fp8 : bf16 ratio)"}}
    del q

    # the same with 128 x 128 weight-block scales (activations per row and
    # 128-wide group)
    qb = wl.make_fp8_weights(spec, device=dev, block=True)

    def fp8_block():
        pkg.moe_forward_fp8(d["hidden"], step.w, step.ids, qb["w13_q"], qb["w2_q"],
                            qb["w13_scale"], qb["w2_scale"], None, None, ws8, step.out)

    ms = max_over_ranks(time_steps(fp8_block, K, W, world) / K, world)
    pkg.profiler_start()
    for _ in range(K):
        fp8_block()
    prof = pkg.profiler_stop()
    us = {k: 1e3 * v[1] / max(v[0], 1) for k, v in prof.items()}
    ach = f1 / (us["gemm1_swiglu_fp8_block"] * 1e-6) / 1e12
    out["fp8_w8a8_block"] = {"ms_per_step": round(ms, 4),
                             "tokens_per_s": round(spec.M * world / (ms / 1e3), 1),
                             "tflops": round(spec.flops() / (ms / 1e3) / 1e12, 1),
                             "kernels_us": {k: round(v, 2) for k, v in us.items()},
                             "roofline": {"kernel": "gemm1_swiglu_fp8_block", "bound": "tensor",
                                          "achieved": round(ach, 1), "peak": round(peak8, 1),
                                          "unit": "TFLOP/s", "frac": round(ach / peak8, 4),
                                          "peak_source": "measured burst bf16 x 2 (nominal fp8 : bf16 ratio)"}}
    del qb, ws8
    return out


def measure_wq(step, spec, K, W, world, pk):
    """Weight-only quantised experts on the same layer, prefill and the
    M = 16 decode: int4 (group 128, zero points), MX FP4 and MX FP6 (E2M3).  Decode is
    bound by the weight bytes: touched experts' codes + scales + zero points,
    plus x, out and logits.  Decode runs the decode GEMMs (weights expanded in
    registers); decode_ms_grouped_gemm is the same call through the grouped
    tensor-core GEMMs."""
    import mixture_experts_ffn_softmax_gb300 as pkg
    d = step.d
    dev = d["hidden"].device
    dspec = wl.SPECS["mixtral_decode"]
    dd = wl.make_moe_inputs(dspec, device=dev, weights=False)
    dw, dids = pkg.moe_route(dd["router_logits"], dspec.top_k, "softmax", True)
    touched = int(torch.unique(dids).numel())
    out = {}
    for fmt, G in (("int4", 128), ("mxfp4", 32), ("mxfp6_e2m3", 32)):
        q = wl.make_wq_weights(spec, fmt, G, device=dev)
        args = (q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"], q["w13_zero"], q["w2_zero"],
                q["group_size"])
        ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                    "separate"), dev)
        y = torch.empty_like(d["hidden"])
        yd = torch.empty_like(dd["hidden"])

        def prefill():
            pkg.moe_forward_wq(d["hidden"], step.w, step.ids, fmt, *args, workspace=ws, out=y)

        def decode():
            pkg.moe_forward_wq(dd["hidden"], dw, dids, fmt, *args, workspace=ws, out=yd)

        ms_p = max_over_ranks(time_steps(prefill, K, W, world) / K, world)
        Kd = max(K, 20)
        ms_d = max_over_ranks(time_steps(decode, Kd, max(W, 3), world) / Kd, world)
        # the same decode call through the grouped tensor-core GEMMs, for context
        pkg.set_wq_decode(False)
        try:
            ms_dg = max_over_ranks(time_steps(decode, Kd, max(W, 3), world) / Kd, world)
        finally:
            pkg.set_wq_decode(True)
        pkg.profiler_start()
        for _ in range(Kd):
            decode()
        prof = pkg.profiler_stop()
        wbytes = sum(t.numel() * t.element_size() for k, t in q.items()
                     if isinstance(t, torch.Tensor)) * touched // spec.E
        dbytes = wbytes + dspec.M * dspec.H * 2 * 2 + dspec.M * dspec.E * 4
        out[f"{fmt}_g{G}"] = {
            "prefill_ms_per_step": round(ms_p, 4),
            "prefill_tokens_per_s": round(spec.M * world / (ms_p / 1e3), 1),
            "prefill_tflops": round(spec.flops() / (ms_p / 1e3) / 1e12, 1),
            "decode_ms_per_step": round(ms_d, 4),
            "decode_ms_grouped_gemm": round(ms_dg, 4),
            "decode_tokens_per_s": round(dspec.M * world / (ms_d / 1e3), 1),
            "decode_weight_bytes": wbytes,
            "decode_hbm_roofline_frac": round(dbytes / (pk["hbm_gbs"] * 1e9) / (ms_d / 1e3), 4),
            "decode_kernels_us": {k: round(1e3 * v[1] / v[0], 2) for k, v in prof.items()},
        }
        del q, ws
    return out


# ------------------------------------------------------- CPU oracle legs --
class _ExpertsF64:
    """Host fp64 copies of just the experts a sample uses, indexable like the
    [E, ...] weight tensor (the oracle reads w[e] only for experts with
    routed rows).  Widening happens here, before any timing."""

    def __init__(self, t, experts):
        self.shape = tuple(t.shape)
        self._w = {int(e): wl.to_f64(t[int(e)]) for e in experts}

    def __getitem__(self, e):
        return self._w[int(e)]


def _sample_tokens(spec, n_small=None):
    """Tokens in the CPU sample.  Each expert the sample touches is widened
    to fp64 on the host (3 H I 8 bytes): when all experts fit in 12 GB the
    sample is 256 tokens for E <= 8 and 128 routed rows otherwise (n_small
    overrides), else as many tokens as keep the touched experts within 6 GB."""
    per_expert = 3 * spec.H * spec.I * 8
    if spec.E * per_expert <= 12e9:
        n = n_small or (256 if spec.E <= 8 else max(1, 128 // spec.top_k))
        return min(spec.M, n)
    return min(spec.M, max(1, int(6e9 // per_expert) // spec.top_k))


def _oracle_inputs(spec, d, n):
    import oracle
    x = wl.to_f64(d["hidden"][:n])
    logits = wl.to_f64(d["router_logits"][:n])
    _, ids, _ = oracle.route(logits, spec.top_k, spec.routing_method, spec.renormalize,
                             spec.k_group, spec.group_count, spec.group_select_mode,
                             spec.routed_scaling_factor)
    experts = np.unique(ids)
    w13 = _ExpertsF64(d["w13"], experts)
    w2 = _ExpertsF64(d["w2"], experts)
    b13 = wl.to_f64(d["w13_bias"]) if d.get("w13_bias") is not None else None
    b2 = wl.to_f64(d["w2_bias"]) if d.get("w2_bias") is not None else None
    return x, logits, w13, w2, b13, b2, experts.size


def cpu_baseline(spec, d, budget_s=15.0, kind="oracle"):
    """Times the CPU oracle (as it stands) on a bounded token sample: the
    whole layer (routing + the experts of each sampled token) in fp64."""
    import oracle
    n = _sample_tokens(spec)
    x, logits, w13, w2, b13, b2, n_exp = _oracle_inputs(spec, d, n)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.moe_layer(x, logits, w13, w2, spec.top_k, spec.routing_method, spec.renormalize,
                         spec.k_group, spec.group_count, spec.group_select_mode,
                         spec.routed_scaling_factor, b13, b2)
        reps += 1
        if time.perf_counter() - t0 > budget_s / 2 or reps >= 3:
            break
    dt = (time.perf_counter() - t0) / reps
    return {"value": round(n / dt, 2), "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": kind,
            "sample": f"{n} of {spec.M} tokens of {spec.name} ({n_exp} experts touched), full "
                      f"routing + {spec.top_k} experts per token in fp64 numpy, {reps} rep(s), "
                      f"{dt:.3f} s each"}


def cpu_baseline_batched(spec, d, budget_s=3.0, n_experts=2):
    """The oracle's batched forward on the valid rows of the first n_experts
    experts (their weights widened to fp64 beforehand)."""
    import oracle
    counts = d["expert_num_tokens"][:n_experts].cpu().numpy()
    xb = wl.to_f64(d["x"][:n_experts])
    rw = wl.to_f64(d["row_weight"][:n_experts])
    ex = range(n_experts)
    w13, w2 = _ExpertsF64(d["w13"], ex), _ExpertsF64(d["w2"], ex)
    w13.shape = (n_experts,) + w13.shape[1:]
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.forward_batched(xb, counts, w13, w2, None, None, rw)
        reps += 1
        if time.perf_counter() - t0 > budget_s / 2 or reps >= 3:
            break
    dt = (time.perf_counter() - t0) / reps
    rows = int(counts.sum())
    return {"value": round(rows / dt, 2), "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"the {rows} valid rows of experts 0..{n_experts - 1} of {spec.E} "
                      f"({spec.name}) in fp64 numpy, {reps} rep(s), {dt:.3f} s each"}


def run_reference(args, world, rank, local):
    if rank != 0:
        return
    if args.workload in wl.BATCHED_SPECS:
        print(json.dumps({"impl": "reference", "unavailable":
                          "the reference arm times the contiguous-layout workloads only"}))
        return
    spec = {**wl.SPECS, **wl.PROFILE_SPECS}[args.workload]
    d = wl.make_moe_inputs(spec, device="cpu")
    import oracle
    n = _sample_tokens(spec, n_small=128)
    x, logits, w13, w2, b13, b2, n_exp = _oracle_inputs(spec, d, n)

    def step():
        oracle.moe_layer(x, logits, w13, w2, spec.top_k, spec.routing_method, spec.renormalize,
                         spec.k_group, spec.group_count, spec.group_select_mode,
                         spec.routed_scaling_factor, b13, b2)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    v = round(n / dt, 2)
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {**workload_config(spec), "parallelism": "cpu oracle, one process"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{n} of {spec.M} tokens per step ({n_exp} experts "
                                       f"touched; fp64 numpy oracle)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral_prefill",
                    choices=sorted(wl.SPECS) + sorted(wl.PROFILE_SPECS) + sorted(wl.BATCHED_SPECS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads of the layer family (decode still runs)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--tiles", default="auto", choices=["auto", "single", "pairs"],
                    help="grouped-GEMM tile shape (default: the library's automatic choice)")
    ap.add_argument("--reduce", default="auto", choices=["auto", "separate", "epilogue_atomic"],
                    help="TopKWeightAndReduce choice (default: the library's AUTO rule)")
    ap.add_argument("--pdl", default="on", choices=["on", "off"],
                    help="programmatic dependent launch between the library's kernels")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    OurStep.reduce = args.reduce
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "ours" and args.tiles != "auto":
        import mixture_experts_ffn_softmax_gb300 as pkg
        pkg.set_gemm_tiles(args.tiles)
    if args.impl == "ours" and args.pdl == "off":
        import mixture_experts_ffn_softmax_gb300 as pkg
        pkg.set_pdl(False)
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    elif args.workload in wl.BATCHED_SPECS:
        run_batched(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
