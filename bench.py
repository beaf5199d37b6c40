#!/usr/bin/env python
"""Benchmark of the quantised routed-MoE layer forward on B300.

Workload (default): the GLM-5.2-shaped layer (H=6144, I=2048, E=256 routed + 1 shared
expert, top-8 of 8 groups keep 4, int4 with an fp16 scale per 32 elements) at decode
batch T=1, one fresh seeded token per step. A step is one whole forward (router,
selection, grouping, gate/up + SwiGLU, down + combine). The timed region is one CUDA
graph replay of K steps; step s reads layer copy s mod C (C identical copies at distinct
addresses, so every step streams its experts from HBM rather than L2) and its own x.

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; expert-weight HBM GB/s vs ~8 TB/s at batch 1/32/2048"
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="glm52_decode_t1")
    p.add_argument("--copies", type=int, default=4)
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--cpu-budget", type=float, default=None,
                   help="seconds of oracle time (cpu_baseline: 20 by default; --impl reference: "
                        "scaled with --steps and --warmup by default)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--fp4-peak", action="store_true", help="measure the dense NVFP4 tensor peak and exit")
    p.add_argument("--path", default="auto", choices=["auto", "gemv", "grouped", "generic"],
                   help="force the expert path (per-format GEMV comparisons)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers


def dist_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def workload_config(wl, world):
    """The keys that name the workload, the same on both arms' lines."""
    spec = wl.layer
    return {"workload": wl.name, "tokens_per_step": wl.tokens, "layer": spec.name,
            "weight_format": spec.weight_format, "act_quant": getattr(spec, "act_quant", "none"),
            "parallelism": f"replicas x{world}"}


def rank_seed_base(rank, steps, warmup):
    """First input seed of this rank: rank r draws seeds base .. base + steps + warmup - 1,
    disjoint from every other rank's (each replica processes its own tokens)."""
    return 1000 * rank * (steps + warmup)


def max_over_ranks(value, world, device):
    """The largest of the ranks' `value` (the slowest rank's time): an all_reduce MAX over
    the default process group when world > 1."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, steps, tokens, seconds):
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's time."""
    return world * steps * tokens / seconds


class ClockSampler:
    """SM clock and clock-event reasons sampled on a background thread while the timed
    region runs (NVML when the Python binding is importable, else `nvidia-smi -lms`)."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "hw_power_brake_slowdown": 0x80, "sw_power_cap": 0x4}

    def __init__(self, index: int, period_s: float = 0.002):
        self.index, self.period = index, period_s
        self.samples, self.reasons = [], set()
        self._stop = threading.Event()
        self.mode, self.max_mhz, self.proc = None, None, None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception:
            self.mode = "smi"

    def _run(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for name, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        else:
            import subprocess
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self.mode == "nvml":
            self.t.join()
        elif self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                    for name, val in zip(names, f[2:]):
                        if val.lower() == "active":
                            self.reasons.add(name)
                except (ValueError, IndexError):
                    pass

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": self.mode}


def source_fingerprint(text):
    """sha256 of CUDA sources with /* */ and // comments, trailing blanks and empty lines
    removed: it changes with any change to the code, not with a comment edit."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    code = [line.split("//", 1)[0].rstrip() for line in text.splitlines()]
    return hashlib.sha256("\n".join(c for c in code if c).encode()).hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from a committed ncu
    capture (profiles/traffic.json), or None when there is none or when the code of the
    kernel's sources (the .cu file and the headers it includes) has changed since the
    capture (their fingerprint no longer matches the recorded one)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        if rec.get("workload") != workload:
            return None
        text = ""
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src)) as f:
                text += f.read() + "\n"
        fp = source_fingerprint(text)
    except (OSError, KeyError, ValueError):
        return None
    return float(rec["bytes_per_launch"]) if fp == rec.get("source_fingerprint") else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], "measured"
    except Exception:
        return 6400.0, "fallback"


def measured_tflops():
    """Dense bf16 (= fp16 kind::f16 rate) tensor peak: the measured burst figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], "measured burst bf16 (kind::f16 runs fp16 at the same rate)"
    except Exception:
        return 1800.0, "fallback"


def measured_fp4_tflops():
    """Dense NVFP4 (E2M1, E4M3 scales per 16) tensor peak: the figure `bench.py --fp4-peak`
    measured with cuBLASLt and recorded in profiles/fp4_peak.json, else the measured bf16
    burst peak times the nominal dense fp4/bf16 ratio (13.5 / 2.25)."""
    try:
        with open(os.path.join(ROOT, "profiles", "fp4_peak.json")) as f:
            d = json.load(f)
        return float(d["fp4_tflops"]), "measured burst nvfp4 (torch._scaled_mm, cuBLASLt)"
    except Exception:
        tf, _ = measured_tflops()
        return tf * 13.5 / 2.25, "measured bf16 burst x nominal fp4/bf16 ratio 6"


def fp4_peak():
    """Time a dense NVFP4 GEMM (8192^3, bf16 output) through torch._scaled_mm: best of 10
    after warm-up, CUDA events. Prints one JSON line."""
    import torch
    n = 8192
    g = torch.Generator(device="cuda").manual_seed(0)
    a = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device="cuda", generator=g)
    b = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device="cuda", generator=g)
    a, b = a.view(torch.float4_e2m1fn_x2), b.view(torch.float4_e2m1fn_x2)
    sa = torch.full((n * n // 16,), 1.0, device="cuda").to(torch.float8_e4m3fn)
    sb = torch.full((n * n // 16,), 1.0, device="cuda").to(torch.float8_e4m3fn)
    f = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    best = None
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1000.0
        best = t if best is None else min(best, t)
    print(json.dumps({"fp4_tflops": 2.0 * n ** 3 / best / 1e12, "shape": [n, n, n],
                      "how": "torch._scaled_mm float4_e2m1fn_x2 x float4_e2m1fn_x2, e4m3 scales per 16, "
                             "bf16 out, best of 10, CUDA events", "torch": torch.__version__,
                      "gpu": torch.cuda.get_device_name()}), flush=True)


def expert_bytes(spec):
    """Stored bytes of one expert: (gate/up, down)."""
    H, I = spec.hidden, spec.inter
    if spec.weight_format == "int4_g32":
        per = lambda n, k: n * (k // 2 + k // 32 * 2)
    elif spec.weight_format == "nvfp4":
        per = lambda n, k: n * (k // 2 + k // 16) + 4
    else:   # per-row int8 / int4 / int2 with an fp32 scale per row
        bits = {"int8_row": 8, "int4_row": 4, "int2_row": 2}[spec.weight_format]
        per = lambda n, k: n * (k * bits // 8 + 4)
    return per(2 * I, H), per(H, I)


# ----------------------------------------------------------------- CPU oracle


def host_cpu():
    """(logical cores, CPU model name) of this host."""
    model = None
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
    except Exception:
        pass
    return os.cpu_count() or 1, model


def oracle_tokens_per_s(spec, arrays, T, budget_s, step0=0, max_tokens=8, threads=None):
    """Time the fp64 oracle on successive steps of the workload until ``budget_s``
    seconds have passed (at least one step). Each step routes all T tokens and runs the
    expert FFNs and the combine for the first min(T, max_tokens) of them (the oracle's
    ``tokens=`` restriction), so a step of a large batch stays a bounded sample (NVFP4
    layers, whose h tensor scale depends on every routed token, run the first
    min(T, max_tokens) tokens as a batch of their own instead). Returns
    (tokens/s over the sampled tokens, steps, threads, seconds, sampled tokens per step).
    ``threads`` caps the BLAS thread pool (None: all of the host's cores)."""
    from oracle.moe_oracle import Layer
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    cores = os.cpu_count() or 1
    use = cores if threads is None else min(threads, cores)
    if threadpool_limits is not None:
        with threadpool_limits(limits=use):
            return _oracle_loop(Layer.from_spec(spec, arrays), spec, T, budget_s, step0, max_tokens, use)
    return _oracle_loop(Layer.from_spec(spec, arrays), spec, T, budget_s, step0, max_tokens, 1)


def _oracle_loop(layer, spec, T, budget_s, step0, max_tokens, threads):
    from synth import make_x
    n = min(T, max_tokens)
    toks = np.arange(n)
    t0 = time.perf_counter()
    steps = 0
    while True:
        x = make_x(spec, T, step0 + steps)
        if spec.weight_format == "nvfp4":
            # the h tensor scale needs every routed h of the batch: sample a T=n batch
            layer.forward(x[:n])
        else:
            layer.forward(x, tokens=toks)
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return steps * n / dt, steps, threads, dt, n


# --------------------------------------------------------------------- arms


def run_reference(args):
    rank, _, world = dist_info()
    if rank != 0:
        return
    from synth import WORKLOADS, make_layer
    wl = WORKLOADS[args.workload]
    spec, T = wl.layer, wl.tokens
    arrays = make_layer(spec)
    budget = (args.cpu_budget if args.cpu_budget is not None
              else min(150.0, max(10.0, 0.15 * (args.steps + args.warmup))))
    if args.warmup:
        oracle_tokens_per_s(spec, arrays, T, 0.0, step0=10_000)
    value, steps, threads, dt, n = oracle_tokens_per_s(spec, arrays, T, budget)
    cores, model = host_cpu()
    sample = (f"fp64 numpy oracle on {threads} of {cores} host threads ({model}), {steps} steps of the "
              f"workload (T={T} routed, expert FFNs and combine for {n} tokens per step), {dt:.1f} s "
              f"time-bounded")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * dt / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(wl, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import quantized_moe_noaux_b300 as moe
    from synth import WORKLOADS, make_layer, make_x

    def x_to_device(x, act_dtype):
        if act_dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    rank, local_rank, world = dist_info()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl")
    wl = WORKLOADS[args.workload]
    spec, T = wl.layer, wl.tokens
    K, W, C = args.steps, args.warmup, max(1, args.copies)
    arrays = make_layer(spec)
    layers = [moe.MoeLayer.from_spec(spec, arrays, max_tokens=T) for _ in range(C)]
    path = {"auto": moe.PATH_AUTO, "gemv": moe.PATH_GEMV, "grouped": moe.PATH_GROUPED,
            "generic": moe.PATH_GENERIC}[args.path]
    for L in layers:
        L.set_path(path)
    stream = torch.cuda.Stream()
    dt = torch.bfloat16 if spec.act_dtype == "bf16" else torch.float32
    H = spec.hidden
    base = rank_seed_base(rank, K, W)     # distinct tokens per rank
    X = torch.stack([x_to_device(make_x(spec, T, base + s), spec.act_dtype) for s in range(K + W)])
    OUT = torch.empty((K + W, T, H), dtype=dt, device="cuda")

    with torch.cuda.stream(stream):
        # warm-up (eager), also the source of per-step unique-expert counts
        uniq = []
        for s in range(W):
            layers[s % C].forward(X[s], OUT[s], stream)
        for s in range(K):
            layers[s % C].forward(X[W + s], OUT[W + s], stream)
            off = layers[s % C].routing(T, stream)["offsets"]
            uniq.append(int(np.count_nonzero(np.diff(off))))
        torch.cuda.synchronize()
        for L in layers:
            assert L.status() == 0, "device status word set"

        launches0 = sum(L.launch_count() for L in layers)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for s in range(K):
                layers[s % C].forward(X[W + s], OUT[W + s], stream)
        launches = sum(L.launch_count() for L in layers) - launches0
        graph.replay()
        torch.cuda.synchronize()

        # timed region
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local_rank) as clocks:
            # a loaded lead-in of untimed replays, so clock samples reflect the same load
            t_end = time.time() + 0.3
            while time.time() < t_end:
                graph.replay()
                torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("timed")   # lets a profiler keep only the timed launches
            ev0.record(stream)
            graph.replay()
            ev1.record(stream)
            torch.cuda.nvtx.range_pop()
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ms = max_over_ranks(ev0.elapsed_time(ev1), world, "cuda")
        value = job_throughput(world, K, T, ms / 1000.0)

        # per-stage durations over a replay of the same K steps (stage events recorded
        # inside a second graph capture)
        for L in layers:
            L.enable_timing((K + C - 1) // C)
        graph2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph2, stream=stream):
            for s in range(K):
                layers[s % C].forward(X[W + s], OUT[W + s], stream)
        graph2.replay()
        torch.cuda.synchronize()
        stage_ms = {name: 0.0 for name in moe.STAGES}
        nfw = 0
        for L in layers:
            st, n = L.stage_times()
            nfw += n
            for kk, v in st.items():
                stage_ms[kk] += v
            L.enable_timing(0)

        # end-to-end through the public API with host buffers (pinned)
        KE = min(args.e2e_steps, K)
        xh = X[W:W + KE].cpu().pin_memory()
        oh = torch.empty((KE, T, H), dtype=dt).pin_memory()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(KE):
            layers[s % C].forward_host(xh[s], oh[s], stream)
        e2e_value = job_throughput(world, KE, T, max_over_ranks(time.perf_counter() - t0, world, "cuda"))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    gu_b, d_b = expert_bytes(spec)
    n_units = sum(u + 1 for u in uniq)                # routed unique + shared, over K steps
    router_b = spec.n_experts * spec.hidden * (4 if spec.router_dtype == "f32" else 2)
    if spec.shared_format == "bf16":                  # separately stored bf16 shared expert
        sh_gu_b, sh_d_b = 2 * spec.inter * spec.hidden * 2, spec.hidden * spec.inter * 2
        n_units -= K
        unit_gu = n_units * gu_b + K * sh_gu_b
        unit_all = n_units * (gu_b + d_b) + K * (sh_gu_b + sh_d_b)
    else:
        unit_gu = n_units * gu_b
        unit_all = n_units * (gu_b + d_b)
    fused = launches == K                              # decode path: one kernel per step
    generic = args.path == "generic" or spec.weight_format.endswith("_row") or \
        getattr(spec, "act_quant", "none") != "none"
    dtype = "f32" if generic else "nvfp4" if spec.weight_format == "nvfp4" else "f16"
    peak_bw, peak_kind = measured_peaks()
    peak_tf, tf_kind = measured_tflops()
    step_s = ms / K / 1000.0
    if fused:
        # one kernel per step: its time per launch is the graph-timed step (the launch
        # overhead included, so this is a lower bound of the kernel's own rate)
        dom_bytes = unit_all + K * router_b
        achieved = dom_bytes / (ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "kernel": "moe_decode_kernel (router, selection, gate/up, down, combine)",
                    "achieved": achieved, "peak": peak_bw, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": achieved / peak_bw, "traffic": recorded_traffic("moe_decode_kernel", wl.name),
                    "bytes_per_launch": dom_bytes / K,
                    "time_per_launch_ms": ms / K, "time_source": "CUDA-graph replay time per step"}
    else:
        # dominant kernel: the routed gate/up GEMM (2/3 of the routed FLOPs and weight bytes;
        # a shared expert in the routed format runs in the same launch, a bf16 one in the
        # next stage)
        dom_s = stage_ms["gate_up_or_fused"] / 1000.0
        if generic:
            kernel = "expert_up_kernel gate/up (CUDA cores, fp32)"
            rows, dom_bytes = T * spec.top_k + T, unit_gu
            peak_t, t_kind = 148 * 128 * 2 * 2.032e9 / 1e12, "fp32 FMA: 148 SMs x 128 lanes x 2 x 2.032 GHz"
        elif spec.weight_format == "nvfp4" and spec.shared_format == "bf16":
            kernel = "moe_gemm_fp4_kernel gate/up (tcgen05 kind::mxf4nvf4)"
            rows, dom_bytes = T * spec.top_k, n_units * gu_b
            peak_t, t_kind = measured_fp4_tflops()
        else:
            kernel = "moe_gemm_kernel gate/up (tcgen05 kind::f16)"
            rows, dom_bytes = T * spec.top_k + T, unit_gu
            peak_t, t_kind = peak_tf, tf_kind
        flops = K * 2.0 * rows * 2 * spec.inter * spec.hidden
        ach_t, ach_b = flops / dom_s / 1e12, dom_bytes / dom_s / 1e9
        tensor = flops / dom_bytes > peak_t * 1e12 / (peak_bw * 1e9)
        roofline = {"bound": "tensor" if tensor else "hbm", "kernel": kernel,
                    "achieved": ach_t if tensor else ach_b, "peak": peak_t if tensor else peak_bw,
                    "peak_kind": t_kind if tensor else peak_kind, "unit": "TFLOP/s" if tensor else "GB/s",
                    "frac": ach_t / peak_t if tensor else ach_b / peak_bw,
                    "traffic": recorded_traffic("moe_gemm_fp4_kernel", wl.name) if "fp4" in kernel else None,
                    "frac_hbm": ach_b / peak_bw, "frac_tensor": ach_t / peak_t,
                    "achieved_gbs": ach_b, "achieved_tflops": ach_t, "hbm_peak": peak_bw,
                    "tensor_peak": peak_t, "tensor_peak_kind": t_kind,
                    "bytes_per_launch": dom_bytes / K, "flops_per_launch": flops / K,
                    "time_per_launch_ms": dom_s * 1000.0 / K,
                    "time_source": "stage events around the launch, CUDA-graph replay"}
        all_flops = K * 2.0 * (T * spec.top_k + T) * 3 * spec.inter * spec.hidden
        roofline["layer_tflops"] = all_flops / (ms / 1000.0) / 1e12
    roofline["step_expert_bytes"] = unit_all / K
    roofline["step_expert_gbs"] = unit_all / K / step_s / 1e9
    roofline["frac_of_8tbs_nominal"] = unit_all / K / step_s / 8e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded, random-init weights)",
            "config": {**workload_config(wl, world),
                       "layer_copies": C, "l2": f"inputs larger than L2: {C} layer copies "
                       "rotated per step, each step streams its experts from HBM",
                       "unique_experts_mean": float(np.mean(uniq)), "path": args.path},
            "roofline": roofline,
            "stage_ms_per_step": {k: v / max(nfw, 1) for k, v in stage_ms.items()},
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": T * H * (2 if spec.act_dtype == "bf16" else 4),
                    "d2h_bytes_per_step": T * H * (2 if spec.act_dtype == "bf16" else 4),
                    "steps": KE}}
    if wl.name.startswith("glm52_mtp_verify"):
        # MTP draft-verify: expert loads of one verify forward, per position and per token
        # generated at the pages' 2.2-2.8 tokens per forward (a decode step loads top_k + 1)
        loads = float(np.mean(uniq)) + 1.0
        line["mtp"] = {"draft": T - 1, "expert_loads_per_forward": loads, "per_position": loads / T,
                       "per_generated_token": {"2.2": loads / 2.2, "2.8": loads / 2.8},
                       "decode_loads_per_token": spec.top_k + 1}
    if world == 1 and not args.no_cpu_baseline:
        cores, model = host_cpu()
        cpu_budget = 20.0 if args.cpu_budget is None else args.cpu_budget
        v, steps, threads, dt_cpu, n = oracle_tokens_per_s(spec, arrays, T, cpu_budget / 2)
        v1, steps1, _, dt1, _ = oracle_tokens_per_s(spec, arrays, T, cpu_budget / 2, threads=1)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "model": model, "value_1_thread": v1,
                                "sample": f"{steps} steps of the workload on {threads} threads ({dt_cpu:.1f} s) "
                                          f"and {steps1} on 1 thread ({dt1:.1f} s), T={T} routed, {n} tokens "
                                          f"through the experts per step, fp64 numpy"}
    print(json.dumps(line), flush=True)
    for L in layers:
        L.close()
    if world > 1:
        dist.destroy_process_group()


def link_h2d_gbs(torch):
    """Pinned host -> device copy bandwidth (1 GiB, best of 5, CUDA events): the host link's
    measured peak, the denominator of the expert cache's link fraction."""
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8).pin_memory()
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1000.0
        best = t if best is None else min(best, t)
    return n / best / 1e9


def run_hostcache(args):
    """Decode through a stack of GLM-shaped int4 layers whose routed experts live in host
    memory, each with an HBM cache of a few expert slots (the pages' engine: experts streamed
    from slower storage into a per-layer LRU cache, router-driven prefetch of the next layer,
    a pinned hot set learned from usage). Token t's input to layer l is drawn correlated with
    its input to layer l - 1 (x_l = rho x_(l-1) + sqrt(1 - rho^2) z), so predicting layer l's
    experts from layer l - 1's input is informative but not exact. Three passes over the same
    tokens: LRU only, LRU + prefetch, LRU + prefetch + the hot set pinned after the first
    pass. Host-synchronous per layer (the host reads the routing back), timed by wall clock."""
    import torch

    import quantized_moe_noaux_b300 as moe
    from synth import WORKLOADS, make_layer

    wl = WORKLOADS[args.workload]
    spec = wl.layer
    n_layers, slots, rho, n_tok = 4, 32, 0.9, min(args.steps, wl.steps)
    arrays = make_layer(spec)
    layers = [moe.MoeLayer.from_spec(spec, arrays, max_tokens=1, cache_slots=slots) for _ in range(n_layers)]
    rng = np.random.default_rng(77)
    xs = np.empty((n_tok, n_layers, spec.hidden), np.float32)
    for t in range(n_tok):
        xs[t, 0] = rng.standard_normal(spec.hidden, dtype=np.float32)
        for l in range(1, n_layers):
            xs[t, l] = rho * xs[t, l - 1] + np.float32(np.sqrt(1 - rho * rho)) * rng.standard_normal(
                spec.hidden, dtype=np.float32)
    xb = torch.from_numpy(xs).to(torch.bfloat16).cuda()
    out = torch.empty((1, spec.hidden), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    link = link_h2d_gbs(torch)

    def one_pass(prefetch):
        for L in layers:
            L.reset_status()
        before = [L.cache_stats() for L in layers]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for t in range(n_tok):
            for l in range(n_layers):
                if prefetch and l + 1 < n_layers:
                    layers[l + 1].prefetch(xb[t, l:l + 1], stream)   # next layer's experts from this input
                layers[l].forward(xb[t, l:l + 1], out, stream)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        after = [L.cache_stats() for L in layers]
        d = {k: sum(a[k] - b[k] for a, b in zip(after, before)) for k in moe.MoeLayer.CACHE_STATS}
        routed = d["hits"] + d["misses"]
        return {"tokens_per_s": n_tok / dt, "ms_per_token": dt * 1000 / n_tok,
                "expert_hit_rate": d["hits"] / max(routed, 1),
                "prefetched": d["prefetched"], "prefetch_hits": d["prefetch_hits"],
                "h2d_gb_per_token": d["bytes_h2d"] / n_tok / 1e9, "link_gbs": d["bytes_h2d"] / dt / 1e9,
                "link_frac": d["bytes_h2d"] / dt / 1e9 / link, "evictions": d["evictions"]}

    one_pass(False)                     # warm-up pass: fills the caches and the usage counts
    lru = one_pass(False)
    pre = one_pass(True)
    for L in layers:
        L.cache_pin_hot(slots - 8)      # keep min(E, T * k) = 8 slots free for the rest
    pin = one_pass(True)
    for L in layers:
        assert L.status() == 0
        L.close()
    line = {"metric": METRIC, "value": pin["tokens_per_s"], "unit": UNIT, "n_gpus": 1, "steps": n_tok,
            "warmup": n_tok, "ms_per_step": pin["ms_per_token"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded, random-init weights)",
            "config": {**workload_config(wl, 1), "layers": n_layers, "cache_slots_per_layer": slots, "experts_per_layer": spec.n_experts,
                       "input_correlation_between_layers": rho,
                       "host_store_gb_per_layer": (2 * spec.inter * spec.hidden + spec.hidden * spec.inter) * 9 / 16
                       * spec.n_experts / 1e9},
            "roofline": {"bound": "host link", "achieved": pin["link_gbs"], "peak": link,
                         "peak_kind": "measured pinned host->device copy (1 GiB)", "unit": "GB/s",
                         "frac": pin["link_frac"], "traffic": None},
            "modes": {"lru": lru, "lru_prefetch": pre, "lru_prefetch_pinned": pin},
            "gpu_launches": None}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.fp4_peak:
        fp4_peak()
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "glm52_hostcache_t1":
        run_hostcache(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
