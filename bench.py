"""Benchmark of the data-parallel collective path on GB300.

A step is one FSDP gradient reduce-scatter over K=8 virtual ranks: eight
64 Mi-element bf16 gradients (N(0, 1e-3), seed = rank) folded in the ring's
order in fp32, scaled by 1/8 and written as eight 8 Mi-element shards in both
fp32 and bf16 -- one call of dp_reduce_scatter_dual.  The metric is algorithmic
HBM bytes (8 x 128 MiB read + 8 x 48 MiB written per step) per second.

Inputs (1 GiB) are larger than L2 (129 MB), so steps run back to back with no
L2 flush.  Timing: W warm-up steps, then K timed steps between CUDA events on
the launching stream, with a barrier and a device synchronize on both sides;
the maximum over ranks is reported.  Under torchrun each rank runs an
independent replica on its own GPU (the virtual ranks never leave one GPU),
so scaling is weak and no collective is on the data path.

At N=1 it also measures the other rows of the path (all-reduce and
all-gather at K=8, the fused all-gather + GEMM, and the variable-length
step) and prints them under "rows".  ``--impl reference`` times the CPU
oracle instead, on bounded samples of the same workload.
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

METRIC = "RS/allreduce HBM GB/s (% of ~8 TB/s peak) at K=8; AG+GEMM TFLOP/s"
MiB = 1 << 20
K_RANKS = 8
N_ELEMS = 64 * MiB
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "ring_allreduce_gradient_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, src_hash):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("source_hash") != src_hash:
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        time.sleep(0.15)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def time_events(fn, reps, stream):
    """Average per-call device time (ms) of fn() over reps, events on `stream`."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    from ring_allreduce_gradient_gb300 import binding as B
    from ring_allreduce_gradient_gb300 import build as cuda_build
    from ring_allreduce_gradient_gb300 import costmodel as cm
    import workloads

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or ws == 1:
        cuda_build.build()
    if ws > 1:
        dist.barrier()
    B.load()
    hbm_peak, bf16_peak, bf16_sus, peak_kind = peaks()

    K, N = K_RANKS, N_ELEMS
    C = N // K
    bufs = workloads.fsdp_grads_device(K, N, dev)
    o32 = [torch.empty(C, dtype=torch.float32, device=dev) for _ in range(K)]
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    step_bytes = cm.reduce_scatter_hbm_bytes(K, N, "bf16", ("f32", "bf16"))

    def step():
        B.dp_reduce_scatter_dual(bufs, K, N, B.DP_BF16, o32, o16, 1.0 / K, sh)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    # timed region
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for a, b in per:
            a.record(stream)
            step()
            b.record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(stop)
    launch_ms = [a.elapsed_time(b) for a, b in per]
    if ws > 1:
        t = torch.tensor([elapsed_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    assert B.dp_get_device_error(sh) == B.DP_OK

    value = step_bytes * args.steps * ws / (elapsed_ms * 1e-3) / 1e9
    avg_launch_ms = statistics.mean(launch_ms)
    achieved = step_bytes / (avg_launch_ms * 1e-3) / 1e9
    src_hash = source_hash("dp_stream.cu", "dp_common.cuh")

    # end to end: pinned host inputs -> device -> the same call -> host outputs
    e2e = None
    if not args.no_e2e:
        hin = [torch.empty(N, dtype=torch.bfloat16, pin_memory=True) for _ in range(K)]
        for h, b in zip(hin, bufs):
            h.copy_(b)
        h32 = [torch.empty(C, dtype=torch.float32, pin_memory=True) for _ in range(K)]
        h16 = [torch.empty(C, dtype=torch.bfloat16, pin_memory=True) for _ in range(K)]

        def e2e_step():
            with torch.cuda.stream(stream):
                for b, h in zip(bufs, hin):
                    b.copy_(h, non_blocking=True)
                step()
                for h, o in zip(h32, o32):
                    h.copy_(o, non_blocking=True)
                for h, o in zip(h16, o16):
                    h.copy_(o, non_blocking=True)

        e2e_steps = max(3, min(args.steps, 20))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b)
        if ws > 1:
            t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_ms = float(t.item())
        e2e = {"value": step_bytes * e2e_steps * ws / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": K * N * 2, "d2h_bytes_per_step": N * 4 + N * 2,
               "ms_per_step": e2e_ms / e2e_steps}
        del hin, h32, h16

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_rs(bufs, args.cpu_sample_mib)

    rows = None
    if ws == 1 and not args.no_rows:
        del o32, o16
        rows = measure_rows(dev, stream, hbm_peak, bf16_peak, peak_kind, args)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": "FSDP gradient reduce-scatter: K=8 virtual ranks x 64Mi bf16 "
                            "N(0,1e-3), ring-order fp32 fold, scale 1/8, fp32+bf16 shards",
                "K": K, "N_per_rank": N, "in_dtype": "bf16", "out_dtypes": ["f32", "bf16"],
                "l2": "inputs 1 GiB per step > 129 MB L2; no flush",
                "parallelism": f"replicas x{ws} (virtual ranks on one GPU each)",
                "algorithmic_bytes_per_step": step_bytes,
            },
            "roofline": {
                "kernel": "rs_vec_kernel<bf16, K=8, fp32+bf16 out>",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "peak_kind": f"{peak_kind} (copy bandwidth, burst)", "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "traffic": ncu_traffic("rs_dual_bf16_k8", src_hash),
                "algorithmic_bytes": step_bytes,
                "avg_launch_ms": avg_launch_ms,
            },
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def cpu_baseline_rs(bufs, sample_mib):
    """The oracle's ring simulator on the first sample_mib Mi elements of
    every rank's gradient (same data), single-threaded on the host."""
    import numpy as np
    import oracle
    import workloads
    from ring_allreduce_gradient_gb300 import costmodel as cm

    K = len(bufs)
    n = min(sample_mib * MiB, bufs[0].numel())
    n -= n % K
    host = [workloads.torch_bf16_to_bits(b[:n]) for b in bufs]
    t0 = time.perf_counter()
    oracle.reduce_scatter(host, 1.0 / K)
    dt = time.perf_counter() - t0
    nbytes = cm.reduce_scatter_hbm_bytes(K, n, "bf16", ("f32", "bf16"))
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"ring step simulator, K={K} ranks x {n} bf16 elements (first "
                      f"{n / bufs[0].numel():.3f} of each rank's 64Mi gradient), one call"}


# ----------------------------------------------------------------------------
# the other rows, measured at N=1 after the headline
# ----------------------------------------------------------------------------

def measure_rows(dev, stream, hbm_peak, bf16_peak, peak_kind, args):
    import torch

    from ring_allreduce_gradient_gb300 import binding as B
    from ring_allreduce_gradient_gb300 import costmodel as cm
    import workloads

    sh = stream.cuda_stream
    rows = {}
    reps = args.row_reps

    def med(xs):
        return statistics.median(xs)

    with torch.cuda.stream(stream):
        # all-reduce, K=8 x 256 MiB fp32 per rank (in place), and x 1 GiB
        for mib in (256, 1024):
            K, N = 8, mib * MiB // 4
            bufs = workloads.sweep_bufs_device(K, N, dev)
            nbytes = cm.all_reduce_hbm_bytes(K, N, "f32")
            fn = lambda: B.dp_ring_allreduce(bufs, K, N, B.DP_FP32, 1.0 / K, sh)
            for _ in range(3):
                fn()
            ms = med(time_events(fn, reps, stream))
            gbs = nbytes / (ms * 1e-3) / 1e9
            rows[f"allreduce_k8_{mib}MiB_f32"] = {
                "ms": ms, "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4),
                "ring_transport_bytes_per_rank": cm.ring_allreduce_bytes_per_rank(N * 4 * 1.0, K)}
            del bufs
            torch.cuda.empty_cache()

        # all-gather, K=8 shards of 32 MiB fp32 -> 8 x 256 MiB
        K, Cg = 8, 32 * MiB // 4
        shards = [torch.randn(Cg, device=dev) for _ in range(K)]
        outs = [torch.empty(K * Cg, device=dev) for _ in range(K)]
        fn = lambda: B.dp_all_gather(shards, K, Cg, B.DP_FP32, outs, sh)
        for _ in range(3):
            fn()
        ms = med(time_events(fn, reps, stream))
        gbs = cm.all_gather_hbm_bytes(K, Cg, "f32") / (ms * 1e-3) / 1e9
        rows["allgather_k8_256MiB_f32"] = {"ms": ms, "GB/s": round(gbs, 1),
                                           "frac_hbm": round(gbs / hbm_peak, 4)}
        del shards, outs
        torch.cuda.empty_cache()

        # fused all-gather + GEMM: (b) x[8192,4096], w_k[512,4096] x 8; (a) fixture
        for name, (M, D, Kw, Fs) in {"agmm_b_8192x4096x4096": (8192, 4096, 8, 512),
                                     "agmm_a_128x512x512": (128, 512, 8, 64)}.items():
            g = torch.Generator(device=dev)
            g.manual_seed(40)
            x = (torch.randn(M, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
            ws_ = [(torch.randn(Fs, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
                   for _ in range(Kw)]
            y = torch.empty(M, Kw * Fs, dtype=torch.bfloat16, device=dev)
            fn = lambda: B.dp_allgather_matmul(x, M, D, ws_, Kw, Fs, y, B.DP_BF16, sh)
            for _ in range(3):
                fn()
            ms = med(time_events(fn, reps, stream))
            tf = cm.gemm_flops(M, Kw * Fs, D) / (ms * 1e-3) / 1e12
            rows[name] = {"ms": ms, "us": ms * 1e3, "TFLOP/s": round(tf, 1),
                          "frac_bf16": round(tf / bf16_peak, 4),
                          "peak": f"{bf16_peak} TFLOP/s bf16 dense ({peak_kind}, burst)"}
            assert B.dp_get_device_error(sh) == B.DP_OK
            del x, ws_, y
        torch.cuda.empty_cache()

        # variable-length step: 32 layers x 16Mi, K=8, fused accumulate+settle,
        # unpadded vs padded, and the two-phase (accumulate kernels + RS) path
        K, N, L = 8, 16 * MiB, args.odc_layers
        m, toks = workloads.odc_schedule(K)
        Mx = max(m)
        grads = [[[workloads.odc_grad(l, r, j, N, int(toks[r, j]), dev) for j in range(m[r])]
                  for r in range(K)] for l in range(L)]
        o32 = [torch.empty(N // K, device=dev) for _ in range(K)]
        o16 = [torch.empty(N // K, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        tables_nopad = [[g for r in range(K) for g in (grads[l][r] + [None] * (Mx - m[r]))]
                        for l in range(L)]

        def odc(pad):
            mm = [Mx] * K if pad else m
            for l in range(L):
                B.dp_odc_reduce_scatter(tables_nopad[l], mm, K, Mx, N, B.DP_BF16, o32, o16,
                                        1.0 / K, sh)

        accs = [torch.empty(N, device=dev) for _ in range(K)]

        def two_phase(pad):
            for l in range(L):
                for r in range(K):
                    last = Mx if pad else m[r]
                    for j in range(last):
                        g = grads[l][r][j] if j < m[r] else None
                        B.dp_grad_accumulate(accs[r], g, N, B.DP_BF16, j == 0, sh)
                B.dp_reduce_scatter_dual(accs, K, N, B.DP_FP32, o32, o16, 1.0 / K, sh)

        total_mb = sum(m)
        res = {}
        for name, fn in (("fused_nopad", lambda: odc(False)), ("fused_pad", lambda: odc(True)),
                         ("two_phase_nopad", lambda: two_phase(False)),
                         ("two_phase_pad", lambda: two_phase(True))):
            fn()
            ms = med(time_events(fn, max(3, reps // 4), stream))
            res[name] = {"ms_per_step": ms}
        fused_bytes = L * cm.odc_fused_hbm_bytes(total_mb, N, "bf16", ("f32", "bf16"))
        gbs = fused_bytes / (res["fused_nopad"]["ms_per_step"] * 1e-3) / 1e9
        res["fused_nopad"]["GB/s"] = round(gbs, 1)
        res["fused_nopad"]["frac_hbm"] = round(gbs / hbm_peak, 4)
        res["pad_over_nopad_fused"] = round(res["fused_pad"]["ms_per_step"] /
                                            res["fused_nopad"]["ms_per_step"], 4)
        res["pad_over_nopad_two_phase"] = round(res["two_phase_pad"]["ms_per_step"] /
                                                res["two_phase_nopad"]["ms_per_step"], 4)
        res["layers"] = L
        res["microbatches_per_rank"] = m
        rows["odc_step_k8_32x16Mi"] = res
        assert B.dp_get_device_error(sh) == B.DP_OK
        del grads, tables_nopad, accs, o32, o16
        torch.cuda.empty_cache()
    return rows


# ----------------------------------------------------------------------------
# the reference arm: the CPU oracle, as it stands
# ----------------------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    import workloads
    from ring_allreduce_gradient_gb300 import costmodel as cm

    oracle.build()
    K = K_RANKS
    n = args.ref_sample_mib * MiB
    host = []
    for r in range(K):
        g = np.random.default_rng(r).standard_normal(n, dtype=np.float32) * np.float32(1e-3)
        host.append(workloads.to_bf16_bits(g))
    nbytes = cm.reduce_scatter_hbm_bytes(K, n, "bf16", ("f32", "bf16"))
    for _ in range(args.warmup):
        oracle.reduce_scatter(host, 1.0 / K)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.reduce_scatter(host, 1.0 / K)
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    sample = (f"ring step simulator, K={K} ranks x {n} bf16 elements per step "
              f"({n / N_ELEMS:.4f} of the 64Mi per-rank gradient), same recipe")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "FSDP gradient reduce-scatter: K=8 virtual ranks x 64Mi bf16 "
                               "N(0,1e-3), ring-order fp32 fold, scale 1/8, fp32+bf16 shards",
                   "K": K, "N_per_rank": N_ELEMS, "sample_N_per_rank": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the other rows' measurements")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--row-reps", type=int, default=20)
    ap.add_argument("--odc-layers", type=int, default=32)
    ap.add_argument("--cpu-sample-mib", type=int, default=16,
                    help="per-rank elements (Mi) of the oracle's timed sample")
    ap.add_argument("--ref-sample-mib", type=int, default=4)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, _, _ = dist_env()
    if ws != args.gpus and not (ws == 1 and args.gpus == 1):
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={ws}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
