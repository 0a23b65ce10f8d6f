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
