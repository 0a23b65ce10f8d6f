"""Host logic of bench.py that needs no GPU: the clock record and the launch
count per forward."""
import bench
from top_routing_grouped_bias_b300 import synth


def _sampler(lines, c0, c1, t0=100.0, t1=100.2):
    s = bench.ClockSampler(0)
    s.lines = [(t0 + 0.01 * (i + 1), ln) for i, ln in enumerate(lines)]
    s.t0, s.t1, s.c0, s.c1 = t0, t1, c0, c1
    return s


def test_clock_record_decodes_mask_and_filters_loaded_samples():
    lines = ["0, 1400, 2032, 1150.0, 0x0000000000000004",   # sw_power_cap
             "0, 1380, 2032, 1160.0, 0x0000000000000004",
             "0, 2032, 2032, 150.0, 0x0000000000000001"]    # idle, below 300 W
    zero = {k: 0.0 for k in bench.ClockSampler.COUNTERS}
    out = _sampler(lines, zero, zero).summary()
    assert out["samples"] == 2 and out["samples_total"] == 3
    assert out["sm_mhz"] == 1390.0 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_record_takes_reasons_from_the_throttle_counters():
    """A 200 ms region in which no sample caught the reason bit but the
    driver's counter advanced by 150 ms: the reason is listed."""
    lines = ["0, 1500, 2032, 1200.0, 0x0000000000000000"] * 3
    c0 = {k: 0.0 for k in bench.ClockSampler.COUNTERS}
    c1 = dict(c0, sw_power_cap=150000.0)
    out = _sampler(lines, c0, c1).summary()
    assert out["throttle_us"]["sw_power_cap"] == 150000
    assert out["reasons"] == ["sw_power_cap"]


def test_launches_per_forward_follow_the_router_plan():
    W = synth.WORKLOADS
    assert bench.kernels_per_forward(W["mixtral_prefill"]) == 7     # split router, one-block dispatch
    assert bench.kernels_per_forward(W["switch_top1"]) == 7         # fused router, fused combine
    assert bench.kernels_per_forward(W["tiny_fp32"]) == 6           # CUDA-core router, one-block dispatch
    assert bench.kernels_per_forward(W["fine_grained_shared"]) == 9  # split router, four-launch dispatch


def _measurement(w, gemm_ms, region_s, mhz):
    import numpy as np
    counts = np.full(w.N, w.T * w.k // w.N)
    return {"counts": counts, "ms": gemm_ms * 1.05, "e2e_ms": gemm_ms * 1.1,
            "staged_ms": gemm_ms * 1.06, "region_s": region_s,
            "stage_ms": {"route": 0.02, "dispatch": 0.03, "grouped_gemm": gemm_ms, "combine": 0.02},
            "clocks": {"sm_mhz": mhz, "sm_max_mhz": 2032.0, "reasons": []}}


def test_roofline_arithmetic_of_the_bench_line():
    """The grouped GEMM's fraction against the burst peak for a short region,
    against the sustained one for a region over 0.5 s, plus the two context
    fractions; a weight-bound batch is held against HBM, with the whole
    layer's fraction beside it."""
    import argparse
    args = argparse.Namespace(steps=10)
    peaks, _ = bench.load_peaks()
    w = synth.WORKLOADS["mixtral_prefill"]
    flops = bench.workload_work(w)["gemm_flops"]
    out = bench.summarize(w, _measurement(w, 2.0, 0.1, 1016.0), args, 1)
    r = out["roofline"]
    achieved = flops / 2.0e-3 / 1e12
    assert r["bound"] == "tensor" and abs(r["achieved"] - achieved) < 0.01
    assert abs(r["frac"] - achieved / peaks["bf16_tflops"]) < 1e-4
    assert abs(r["frac_of_sustained"] - achieved / peaks["bf16_tflops_sustained"]) < 1e-4
    # half the maximum clock: the burst peak scaled by 0.5
    assert abs(r["frac_of_burst_at_sampled_clock"] - 2 * r["frac"]) < 1e-3
    long = bench.summarize(w, _measurement(w, 2.0, 1.0, 1016.0), args, 1)["roofline"]
    assert abs(long["frac"] - achieved / peaks["bf16_tflops_sustained"]) < 1e-4
    assert out["tokens_per_s"] == round(w.T * 10 / (2.1 * 10 / 1e3), 1)
    # decode: about 4 rows per expert, weight-bandwidth bound
    wd = synth.WORKLOADS["mixtral_decode"]
    dec = bench.summarize(wd, _measurement(wd, 0.45, 0.03, 2032.0), args, 1)
    gb = bench.gemm_bytes(wd, _measurement(wd, 0.45, 0.03, 2032.0)["counts"])
    assert dec["roofline"]["bound"] == "hbm"
    assert abs(dec["roofline"]["frac"] - gb / 0.45e-3 / 1e9 / peaks["hbm_gbs"]) < 1e-4
    assert "layer_hbm" in dec and dec["layer_hbm"]["frac"] < dec["roofline"]["frac"]
