"""Host-side pieces of the measurement harness, without a GPU: the clock
summary keeps only the samples stamped inside the timed region, the DRAM
traffic is reported only while the kernel source matches its capture, the
throughput is whole-job work over the slowest rank's time, and the rows'
summary ends with the 4(b) GEMM and stays small enough to survive a reader
that keeps only the end of the output."""
import datetime
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(t, sm, reason_cap="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return (f"{ts}, 0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, "
            f"{reason_cap}")


def test_clock_summary_keeps_the_samples_inside_the_region():
    c = bench.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now, now + 0.1
    c.lines = [_line(now - 0.2, 1200), _line(now + 0.03, 2070), _line(now + 0.06, 2040, "Active"),
               _line(now + 0.5, 1100), "garbage"]
    s = c.summary()
    assert s["samples"] == 2 and s["samples_total"] == 4
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_falls_back_to_the_first_sample_after_the_start():
    c = bench.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now, now + 0.01
    c.lines = [_line(now - 0.3, 1000), _line(now + 0.08, 2060), _line(now + 0.2, 1500)]
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] == 2060.0
    c.lines = []
    assert c.summary()["samples"] == 0


def test_traffic_only_for_the_captured_source():
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    entries = {}
    with open(path) as f:
        for line in f:
            parts = line.split("#", 1)[0].split()
            if len(parts) >= 3:
                entries[parts[0]] = (parts[1], int(parts[2]))
    assert "rs_dual_bf16_k8" in entries
    key, (h, n) = "rs_dual_bf16_k8", entries["rs_dual_bf16_k8"]
    assert bench.ncu_traffic(key, h) == n
    assert bench.ncu_traffic(key, "0" * 16) is None
    assert bench.ncu_traffic("no_such_kernel", h) is None
    # the headline's capture matches the committed kernel sources
    assert bench.source_hash("dp_stream.cu", "dp_stream_common.cuh", "dp_common.cuh") == h


def test_aggregate_rate_is_whole_job_work_over_the_slowest_time():
    # 1.476e9 B per step, 200 steps, 2 ranks, 100 ms for the slowest rank
    v = bench.aggregate_rate(1.476e9, 200, 2, 100.0, 1e9)
    assert abs(v - 1.476e9 * 400 / 0.1 / 1e9) < 1e-6


def test_rows_summary_is_small_and_ends_with_the_gemm():
    rows = {
        "cpu_oracle": {"allreduce_k4_4096_ints_us": 25.0, "sample": "x" * 500},
        "allreduce_sweep": {f"K{K}_{b}": {"K": K, "bytes_per_rank": b, "allreduce_frac": 0.9,
                                          "allreduce_frac_clean_l2": 1.0}
                            for K in (2, 4, 8) for b in (4096, 64 << 20, 256 << 20, 1 << 30)},
        "ag_bulk_copy": {"frac_hbm": 0.98}, "ddp1": {"frac_hbm": 0.87,
                                                     "overlap_mode_frac_hbm": 0.93},
        "agmm_a": {"ms": 0.0102, "graph_us": 5.8},
        "tp_ar": {"frac_bf16": 0.59, "warm_frac_bf16": 0.6},
        "agmm_b_sustained": {"TFLOP/s": 1580.0, "frac_bf16_sustained": 0.9,
                             "clocks": {"sm_mhz": 1950.0, "reasons": ["sw_power_cap"]}},
        "agmm_b": {"TFLOP/s": 1600.0, "frac_bf16": 0.83, "warm_frac_bf16": 0.86,
                   "clean_l2_frac_bf16": 0.85, "warm_TFLOP/s": 1670.0, "ms": 0.171},
    }
    cpu = {"value": 1.5, "threaded": {"value": 13.0, "cores": 16}}
    s = bench.rows_summary(rows, cpu)
    assert list(s)[-1] == "agmm_b"
    assert s["agmm_a_graph_us"] == 5.8 and s["ddp1_overlap_mode_frac"] == 0.93
    assert "sample" not in s["cpu_oracle_rows"]
    assert len(json.dumps(s)) < 2000
    assert bench.rows_summary(None, None) == {"rows": "not measured"}
