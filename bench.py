#!/usr/bin/env python3
"""Benchmark of the MoE-layer forward on B300: tokens/s of one moe_forward per
step on a fixed synthetic batch, the grouped-GEMM roofline fraction, the
end-to-end rate through the C ABI with host buffers, and the CPU oracle timed
on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--configs all|none]

The line's value, config and roofline are those of --workload (default: the
Mixtral-shaped prefill). Its "configs" block repeats the measurement for every
named workload: tokens/s and ms per step, the grouped GEMM against the tensor
peak (or HBM when the batch is weight-bandwidth bound), route / dispatch /
combine against HBM, and the clocks of each region. Stage times come from
events recorded between the four stage calls inside one continuous loop of K
staged steps, so they add up to that loop's step.

N > 1 runs under torchrun, one replica per GPU (tokens are independent, so
every rank runs its own batch with its own copy of the weights and no
collective touches the data path); the timing is the max over ranks.
Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from top_routing_grouped_bias_b300 import api, synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s; grouped-GEMM TFLOP/s & HBM GB/s vs B300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
def kernels_per_forward(w) -> int:
    """Launches of one moe_forward: route 1 (one GEMM with the top-k in its
    epilogue, or the CUDA-core kernel) or 2 (split logits GEMM + selection,
    when the batch has too few 128-token tiles to fill the GPU), dispatch 2
    (one block for count, scan and permute on small batches, plus the gather)
    or 4, grouped GEMM 2, combine 1 (top-1 without a shared expert: the
    combine happens in the down pass)."""
    route = 1
    if w.dtype == "bf16" and w.N <= 256:
        tiles = (w.T + 127) // 128
        kb_total = (w.d + 63) // 64
        s = max(1, min(148 // tiles if tiles else 1, max(1, kb_total // 4)))
        kb_per = (kb_total + s - 1) // s
        if (kb_total + kb_per - 1) // kb_per > 1:
            route = 2
    small = w.T * w.k <= 16384 and ((w.T + 31) // 32) * w.N <= 8192
    dispatch = 2 if small else 4
    combine = 0 if (w.k == 1 and w.F_sh == 0) else 1
    return route + dispatch + 2 + combine


# ------------------------------------------------------------ host logic ---
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar (timing only; no data-path collective)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    return units_per_rank * world / max_seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_work(w):
    """Algorithmic FLOPs and bytes of one forward (touched experts only)."""
    e = 4 if w.dtype == "f32" else 2
    R = w.T * w.k
    gemm_flops = 2.0 * 3 * w.d * w.F * R + 2.0 * 3 * w.d * w.F_sh * w.T
    router_flops = 2.0 * w.N * w.d * w.T
    return dict(gemm_flops=gemm_flops, router_flops=router_flops, R=R, e=e)


def gemm_bytes(w, counts):
    """Algorithmic HBM bytes of the grouped GEMM pair: each touched expert's
    weights once, activations in and out once per pass."""
    e = 4 if w.dtype == "f32" else 2
    touched = int((np.asarray(counts) > 0).sum())
    R = w.T * w.k
    b = touched * 3 * w.d * w.F * e
    b += R * (w.d + w.F) * e + R * (w.F + w.d) * e
    if w.F_sh:
        b += 3 * w.d * w.F_sh * e + w.T * (w.d + w.F_sh) * e * 2
    return b


def traffic_from_profile(workload: str):
    """DRAM traffic per grouped-GEMM stage from the committed ncu summary, or
    None when the summary is missing or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", f"grouped_gemm_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p, encoding="utf-8").read()
    m = re.search(r"dram_bytes_per_stage:\s*([0-9.eE+]+)", txt)
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{16,64})", txt)
    if not m or not h:
        return None
    src = os.path.join(ROOT, "top_routing_grouped_bias_b300", "csrc", "grouped_gemm.cu")
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if not cur.startswith(h.group(1)):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock / power / throttle samples taken while the timed region
    runs, plus the driver's cumulative throttle-time counters read before and
    after it."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active")
    # bits of clocks_event_reasons.active (NVML clocks-event reason mask)
    BITS = ((0x1, "gpu_idle"), (0x2, "applications_clocks_setting"), (0x4, "sw_power_cap"),
            (0x8, "hw_slowdown"), (0x10, "sync_boost"), (0x20, "sw_thermal_slowdown"),
            (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"),
            (0x100, "display_clock_setting"))
    COUNTERS = ("sw_power_cap", "sw_thermal_slowdown", "hw_thermal_slowdown",
                "hw_power_brake_slowdown", "sync_boost")

    def __init__(self, gpu_index: int, interval_ms: int = 10):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self._t = None
        self.c0 = self.c1 = None
        self.t0 = self.t1 = None

    def _counters(self):
        q = ",".join(f"clocks_event_reasons_counters.{c}" for c in self.COUNTERS)
        try:
            r = subprocess.run(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                "-i", str(self.gpu)], capture_output=True, text=True, timeout=10)
            vals = [float(v) for v in r.stdout.strip().split(",")]
            return dict(zip(self.COUNTERS, vals)) if len(vals) == len(self.COUNTERS) else None
        except (OSError, ValueError, subprocess.TimeoutExpired):
            return None

    def __enter__(self):
        self.c0 = self._counters()
        try:
            self.proc = subprocess.Popen(
                ["stdbuf", "-oL", "nvidia-smi", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-i", str(self.gpu), "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *a):
        self.t1 = time.time()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)
        self.c1 = self._counters()

    def summary(self):
        rows = []
        for t, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 5 or not (self.t0 <= t <= self.t1):
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 mask=int(parts[4], 16)))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        # samples taken while the GPU draws well above idle power
        loaded = [r for r in rows if r["power"] > 300] or rows
        reasons = set()
        for r in loaded:
            for bit, name in self.BITS:
                if r["mask"] & bit and bit != 0x1:
                    reasons.add(name)
        out = {"sm_mhz": float(np.median([r["sm"] for r in loaded])),
               "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
               "samples": len(loaded), "samples_total": len(rows),
               "power_w_max": max(r["power"] for r in rows),
               "power_w_median_loaded": float(np.median([r["power"] for r in loaded]))}
        if self.c0 is not None and self.c1 is not None:
            # microseconds the driver spent in each throttle reason during the region
            out["throttle_us"] = {k: round(self.c1[k] - self.c0[k]) for k in self.COUNTERS}
            out["region_s"] = round(self.t1 - self.t0, 3)
            # a reason whose counter advanced by more than 1% of the region was
            # active even if no 10 ms sample caught its bit
            for k, us in out["throttle_us"].items():
                if us > 0.01 * out["region_s"] * 1e6 and k not in out["reasons"]:
                    out["reasons"] = sorted(out["reasons"] + [k])
        return out


# --------------------------------------------------------- CPU baseline ---
def oracle_sample(w, n_tokens: int, seed: int = 0):
    """Inputs of a bounded sample of the workload for the CPU oracle: the
    workload's own weights (drawn with the same generator as the GPU run) and
    its first n_tokens tokens."""
    inp = synth.make_inputs(w, seed=seed, device="cuda" if torch.cuda.is_available() else "cpu")
    f32 = lambda t: None if t is None else t.float().cpu().numpy()
    s = dict(h=f32(inp["h"][:n_tokens]), W_r=f32(inp["W_r"]), W_gate=f32(inp["W_gate"]),
             W_up=f32(inp["W_up"]), W_down=f32(inp["W_down"]), sel_bias=f32(inp["sel_bias"]))
    s["shared"] = None
    if w.F_sh > 0:
        s["shared"] = (f32(inp["Ws_gate"]), f32(inp["Ws_up"]), f32(inp["Ws_down"]))
    del inp
    if torch.cuda.is_available():
        torch.cuda.empty_cache()
    return s


def run_oracle(w, s):
    from oracle import moe_oracle as O
    return O.moe_forward(s["h"], s["W_r"], s["W_gate"], s["W_up"], s["W_down"], w.k, w.score,
                         w.norm, s["sel_bias"], shared=s["shared"])


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


SAMPLE_TOKENS = {"tiny_fp32": 64, "mixtral_prefill": 96, "mixtral_decode": 16,
                 "fine_grained_shared": 24, "switch_top1": 2048}


def cpu_baseline(w, steps: int = 1):
    n = min(w.T, SAMPLE_TOKENS.get(w.name, 64))
    s = oracle_sample(w, n)
    t0 = time.perf_counter()
    for _ in range(steps):
        run_oracle(w, s)
    dt = time.perf_counter() - t0
    return {"value": n * steps / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} of {w.T} tokens of {w.name} (all {w.N} experts' weights), fp64 numpy, "
                      f"{steps} step(s), {dt:.2f} s"}


# ------------------------------------------------------------ our arm ---
def stage_bytes(w):
    """Algorithmic HBM bytes of the memory-bound stages of one forward, from
    the per-token figures: route d*e + 8k (+ the router weight once),
    dispatch d*e + k*d*e + 8k, combine k*d*e + d*e + 4k (+ d*e for the
    shared expert's rows)."""
    e = 4 if w.dtype == "f32" else 2
    T, d, N, k = w.T, w.d, w.N, w.k
    return {"route": T * (d * e + 8 * k) + N * d * e,
            "dispatch": T * (d * e + k * d * e + 8 * k),
            "combine": T * (k * d * e + d * e + 4 * k) + (T * d * e if w.F_sh else 0)}


def measure_workload(args, w, dev, world, local, barrier, headline: bool):
    """Times one workload: K moe_forward steps (the step), K staged steps
    (route, dispatch, expert FFN, combine through their entry points, with
    events between the stages inside one continuous loop), and K steps
    through the public API with host buffers. Returns the raw figures."""
    cfg = api.config_for(w)
    inp = synth.make_inputs(w, seed=0, device=dev)
    tdt = w.torch_dtype
    ws = api.alloc_workspace(cfg, dev)
    outs = api.alloc_outputs(cfg, dev, tdt, logits=False)
    stream = torch.cuda.current_stream(dev)
    K = args.steps

    for _ in range(args.warmup):
        api.forward(cfg, inp, outs, ws, stream)
    torch.cuda.synchronize(dev)
    assert api.read_status(ws) == api.MOE_OK

    # ---- the step: K moe_forward calls, device-resident inputs ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(K):
            api.forward(cfg, inp, outs, ws, stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms = ev0.elapsed_time(ev1) / K
    assert api.read_status(ws) == api.MOE_OK
    counts = outs["counts"].cpu().numpy()

    # ---- the same layer as its four stage calls, events between them ----
    R = w.T * w.k
    idx, gate = outs["idx"], outs["gate"]
    st = {n: torch.empty(sz, dtype=torch.int32, device=dev) for n, sz in
          (("counts", (w.N,)), ("offsets", (w.N + 1,)), ("row_token", (R,)), ("inv", (R,)))}
    x_disp = torch.empty((R, w.d), dtype=tdt, device=dev)
    y_rows = torch.empty((R, w.d), dtype=tdt, device=dev)
    y_sh = torch.empty((w.T, w.d), dtype=tdt, device=dev) if w.F_sh else None
    out2 = torch.empty((w.T, w.d), dtype=tdt, device=dev)
    stages = (
        ("route", lambda: api.moe_route(cfg, inp["h"], inp["W_r"], None, inp["sel_bias"], None,
                                        None, idx, gate, ws, stream)),
        ("dispatch", lambda: api.moe_dispatch(cfg, inp["h"], idx, st["counts"], st["offsets"],
                                              st["row_token"], st["inv"], x_disp, ws, stream)),
        ("grouped_gemm", lambda: api.moe_expert_ffn(
            cfg, x_disp, st["offsets"], inp["W_gate"], inp["W_up"], inp["W_down"], y_rows,
            inp["h"], inp.get("Ws_gate"), inp.get("Ws_up"), inp.get("Ws_down"), y_sh, ws,
            stream)),
        ("combine", lambda: api.moe_combine(cfg, y_rows, st["inv"], gate, y_sh, out2, stream)),
    )
    for _ in range(3):
        for _, fn in stages:
            fn()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
           for _ in range(K)]
    torch.cuda.synchronize(dev)
    t_region = time.perf_counter()
    for i in range(K):
        evs[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            evs[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    region_s = time.perf_counter() - t_region
    assert api.read_status(ws) == api.MOE_OK
    stage_ms = {name: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) / K
                for j, (name, _) in enumerate(stages)}
    staged_ms = evs[0][0].elapsed_time(evs[K - 1][-1]) / K

    # ---- end to end through the public API with host buffers ----
    # Every step copies its hidden states from pinned host memory and its
    # output back; the copies of neighbouring steps overlap the compute.
    h_hosts = [inp["h"].cpu().pin_memory() for _ in range(2)]
    out_hosts = [torch.empty((w.T, w.d), dtype=tdt).pin_memory() for _ in range(2)]
    weights = {k_: v for k_, v in inp.items() if k_ != "h"}
    pipe = api.HostPipeline(cfg, weights, tdt, dev)
    for i in range(max(1, args.warmup)):
        pipe.step(i, h_hosts[i % 2], out_hosts[i % 2])
    pipe.drain()
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.compute)
    pipe.copy_in.wait_event(e0)   # the first copy of the timed region starts after e0
    for i in range(K):
        pipe.step(i, h_hosts[i % 2], out_hosts[i % 2])
    pipe.drain()
    e1.record(pipe.compute)
    torch.cuda.synchronize(dev)
    barrier()
    assert api.read_status(pipe.ws) == api.MOE_OK
    e2e_ms = e0.elapsed_time(e1) / K
    io = {"h2d_bytes_per_step": int(h_hosts[0].numel() * h_hosts[0].element_size()),
          "d2h_bytes_per_step": int(out_hosts[0].numel() * out_hosts[0].element_size())}
    del pipe, h_hosts, out_hosts

    next_rows = None
    if headline:
        def stage_time(fn, reps):
            for _ in range(3):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / reps
        next_rows = time_next_rows(w, cfg, inp, ws, stream, dev, stage_time)
    del inp, ws, outs, st, x_disp, y_rows, y_sh, out2
    torch.cuda.empty_cache()
    return {"ms": max_over_ranks(ms, world, dev),
            "e2e_ms": max_over_ranks(e2e_ms, world, dev),
            "stage_ms": {k_: max_over_ranks(v, world, dev) for k_, v in stage_ms.items()},
            "staged_ms": max_over_ranks(staged_ms, world, dev), "region_s": region_s,
            "counts": counts, "clocks": clk.summary(), "io": io, "next_rows": next_rows}


def summarize(w, m, args, world):
    """Per-workload figures of the bench line: rates, the grouped GEMM's
    roofline, the memory-bound stages against HBM, clocks."""
    peaks, peak_src = load_peaks()
    counts = m["counts"]
    work = workload_work(w)
    gb = gemm_bytes(w, counts)
    gemm_ms = m["stage_ms"]["grouped_gemm"]
    gemm_tflops = work["gemm_flops"] / (gemm_ms * 1e-3) / 1e12
    gemm_gbs = gb / (gemm_ms * 1e-3) / 1e9
    touched = max(1, int((counts > 0).sum()))
    tensor_bound = w.T * w.k / touched >= 64
    # a region of well under a second runs at burst clocks; a longer one
    # settles under the power cap (sustained peak)
    sustained = m["region_s"] > 0.5
    if tensor_bound:
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        if w.dtype == "f32":
            peak = peak / 2.0   # tf32 nominal dense rate is half of bf16
        roof = {"bound": "tensor", "achieved": round(gemm_tflops, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(gemm_tflops / peak, 4),
                "hbm_frac": round(gemm_gbs / peaks["hbm_gbs"], 4)}
    else:
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(gemm_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gemm_gbs / peak, 4),
                "tensor_tflops": round(gemm_tflops, 2)}
    roof.update({"traffic": traffic_from_profile(w.name),
                 "kernel": "grouped GEMM pair (gate/up SwiGLU + down), one moe_expert_ffn call",
                 "algorithmic_flops": work["gemm_flops"], "algorithmic_bytes": gb,
                 "avg_ms": round(gemm_ms, 4),
                 "peak_source": f"{peak_src} ({'sustained' if sustained else 'burst'})"})
    mhz, max_mhz = m["clocks"].get("sm_mhz"), m["clocks"].get("sm_max_mhz")
    if roof["bound"] == "tensor" and mhz and max_mhz:
        # context only: the burst peak scaled to the median SM clock sampled
        # in the timed region (under the power cap the clock sets the rate)
        burst = peaks["bf16_tflops"] / (2.0 if w.dtype == "f32" else 1.0)
        roof["sampled_sm_mhz"] = mhz
        roof["frac_of_burst_at_sampled_clock"] = round(gemm_tflops / (burst * mhz / max_mhz), 4)
    if roof["bound"] == "tensor":
        # context only: against the cuBLAS rate held for seconds under the cap
        sust = peaks["bf16_tflops_sustained"] / (2.0 if w.dtype == "f32" else 1.0)
        roof["frac_of_sustained"] = round(gemm_tflops / sust, 4)
    sb = stage_bytes(w)
    stages = {}
    for name in ("route", "dispatch", "grouped_gemm", "combine"):
        t = m["stage_ms"][name]
        stages[name] = {"ms": round(t, 4)}
        if name in sb:
            gbs = sb[name] / (t * 1e-3) / 1e9
            stages[name].update({"bytes": sb[name], "GB/s": round(gbs, 1),
                                 "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)})
    out = {"tokens_per_s": round(aggregate_rate(w.T * args.steps, world,
                                                m["ms"] * args.steps / 1e3), 1),
           "ms_per_step": round(m["ms"], 4),
           "e2e_tokens_per_s": round(aggregate_rate(w.T * args.steps, world,
                                                    m["e2e_ms"] * args.steps / 1e3), 1),
           "shape": {"T": w.T, "d": w.d, "N": w.N, "ffn": w.F, "k": w.k, "ffn_shared": w.F_sh,
                     "score": w.score, "norm": w.norm, "dtype": w.dtype},
           "roofline": roof, "stages": stages,
           "staged_step_ms": round(m["staged_ms"], 4),
           "load": {"rows_max_over_mean": round(float(counts.max()) / max(1e-9, float(counts.mean())), 3),
                    "idle_experts": int((counts == 0).sum()), "experts": int(w.N)},
           "clocks": m["clocks"]}
    if w.k == 1 and w.F_sh == 0:
        out["note"] = ("moe_forward fuses the combine into the down pass; the staged steps "
                       "run it as a separate launch")
    if not tensor_bound:
        # weight-bandwidth-bound batch: the whole layer against HBM
        layer_b = gb + sb["route"] + sb["dispatch"] + sb["combine"]
        out["layer_hbm"] = {"bytes": layer_b,
                            "GB/s": round(layer_b / (m["ms"] * 1e-3) / 1e9, 1),
                            "frac": round(layer_b / (m["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    return out


def bench_ours(args, w):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    api.load()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    m = measure_workload(args, w, dev, world, local, barrier, headline=True)
    configs = {w.name: summarize(w, m, args, world)}
    if args.configs == "all":
        for name, wc in synth.WORKLOADS.items():
            if name != w.name:
                configs[name] = summarize(wc, measure_workload(args, wc, dev, world, local, barrier,
                                                               headline=False), args, world)
    if rank != 0:
        return None
    head = configs[w.name]
    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) hidden, N(0,std) weights; no dataset)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "ffn": w.F, "k": w.k,
                   "ffn_shared": w.F_sh, "score": w.score, "norm": w.norm,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (expert weights %.2f GB per step)"
                         % (3 * w.N * w.d * w.F * (4 if w.dtype == 'f32' else 2) / 1e9)},
        "roofline": head["roofline"],
        "stages_ms": {k_: v["ms"] for k_, v in head["stages"].items()},
        "staged_step_ms": head["staged_step_ms"],
        "next_rows": m["next_rows"],
        "load": head["load"],
        "gpu_launches": kernels_per_forward(w) * args.steps,
        "e2e": {"value": head["e2e_tokens_per_s"], "unit": "tokens/s", **m["io"]},
        "clocks": head["clocks"],
        "configs": configs,
    }
    return line


def time_next_rows(w, cfg, inp, ws, stream, dev, stage_ms, reps=10):
    """Device time of the rows beyond the core layer on the same batch:
    routing statistics, group-limited routing, the layer with an expert
    capacity (factor 1.25) and the layer with expert-choice routing."""
    peaks, _ = load_peaks()
    T, N, k = w.T, w.N, w.k
    out = {}
    logits = torch.empty((T, N), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    api.moe_route(cfg, inp["h"], inp["W_r"], None, inp["sel_bias"], None, logits, idx, gate, ws,
                  stream)
    stats = torch.empty(3 + 2 * N, dtype=torch.float32, device=dev)
    ms = stage_ms(lambda: api.moe_route_stats(cfg, logits, idx, stats, ws, stream), reps)
    by = T * N * 4 + T * k * 4
    out["route_stats"] = {"ms": round(ms, 4), "GB/s": round(by / ms / 1e6, 1),
                          "hbm_frac": round(by / ms / 1e6 / peaks["hbm_gbs"], 3)}
    ng = next((g for g in (8, 4, 2) if N % g == 0 and (N // g) * (g // 2) >= k), 0)
    if ng:
        grp = api.make_group_config(ng, ng // 2, "topm_sum", min(2, N // ng))
        ms = stage_ms(lambda: api.moe_route_grouped(cfg, grp, inp["h"], inp["W_r"], None,
                                                    inp["sel_bias"], None, logits, idx, gate, ws,
                                                    stream), reps)
        out["route_grouped"] = {"ms": round(ms, 4), "groups": f"{ng} keep {ng // 2} top-2 sum"}
    tdt = w.torch_dtype
    outs = api.alloc_outputs(cfg, dev, tdt, logits=False)
    C = api.expert_capacity(T, k, N, 1.25)
    ms = stage_ms(lambda: api.forward_capacity(cfg, C, inp, outs, ws, stream), reps)
    out["forward_capacity_1.25"] = {"ms": round(ms, 4), "tokens/s": round(T / ms * 1e3, 1),
                                    "capacity": C}
    C = T * k // N
    y = torch.empty((T, w.d), dtype=tdt, device=dev)
    ms = stage_ms(lambda: api.forward_expert_choice(cfg, C, inp, y, ws, stream=stream), reps)
    out["forward_expert_choice"] = {"ms": round(ms, 4), "tokens/s": round(T / ms * 1e3, 1),
                                    "capacity": C}
    assert api.read_status(ws) == api.MOE_OK
    return out


def bench_reference(args, w):
    """The CPU oracle as the reference arm, on bounded samples of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    n = min(w.T, SAMPLE_TOKENS.get(w.name, 64))
    s = oracle_sample(w, n)
    for _ in range(args.warmup):
        run_oracle(w, s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle(w, s)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    sample = f"{n} of {w.T} tokens of {w.name} per step, fp64 numpy oracle"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "ffn": w.F, "k": w.k,
                   "ffn_shared": w.F_sh, "score": w.score, "norm": w.norm},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mixtral_prefill",
                    choices=list(synth.WORKLOADS) + list(synth.PROFILE_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="also time the other named workloads (the 'configs' block)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    w = {**synth.WORKLOADS, **synth.PROFILE_WORKLOADS}[args.workload]
    if args.impl == "reference":
        line = bench_reference(args, w)
    else:
        line = bench_ours(args, w)
        if line is not None:
            line["cpu_baseline"] = None if args.no_cpu_baseline else cpu_baseline(w)
    rank, world, _ = dist_env()
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
