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


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(work_per_step: float, steps: int, world: int, elapsed_ms: float,
                   unit: float) -> float:
    """Whole-job throughput: the work all ranks did over the slowest rank's time."""
    return work_per_step * steps * world / (elapsed_ms * 1e-3) / unit


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
    """Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) from
    the committed ncu summary, if it was captured on the current kernel
    source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split("#", 1)[0].split()
                if len(parts) >= 3 and parts[0] == kernel_key:
                    return int(parts[2]) if parts[1] == src_hash else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from just
    before the timed region to just after it; `mark()` brackets the region,
    and the summary keeps the samples stamped inside it (nvidia-smi takes a
    moment to start, so the sampler starts early and its first samples see
    the GPU idle)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.t1 = time.time()
        time.sleep(0.1)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        import datetime
        rows = []
        for line in list(self.lines):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        # the samples stamped inside the region (20 ms of slack for the
        # timestamps' resolution), else the first one after its start, else
        # every sample
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 - 0.02 <= r[0] <= self.t1 + 0.02]
        after = [r for r in rows if self.t0 is not None and r[0] >= self.t0 - 0.02][:1]
        use = inside or after or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for r in use for n, v in zip(names, r[3]) if v.lower() == "active"}
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": use[-1][2],
                "reasons": sorted(reasons), "samples": len(inside),
                "samples_total": len(rows)}


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
# workloads: each returns the step closure and its algorithmic cost
# ----------------------------------------------------------------------------

def make_workload(name, dev, sh, odc_layers=32, ar_mib=1024):
    import torch

    from ring_allreduce_gradient_gb300 import binding as B
    variant = B.dp_get_collective_variant()
    from ring_allreduce_gradient_gb300 import costmodel as cm
    import workloads

    if name == "rs":
        K, N = K_RANKS, N_ELEMS
        C = N // K
        bufs = workloads.fsdp_grads_device(K, N, dev)
        o32 = [torch.empty(C, dtype=torch.float32, device=dev) for _ in range(K)]
        o16 = [torch.empty(C, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        return dict(
            step=lambda: B.dp_reduce_scatter_dual(bufs, K, N, B.DP_BF16, o32, o16, 1.0 / K, sh),
            bytes=cm.reduce_scatter_hbm_bytes(K, N, "bf16", ("f32", "bf16")), bound="hbm",
            kernel="rs_vec_kernel<bf16, K=8, fp32+bf16 out>", traffic_key="rs_dual_bf16_k8",
            src=("dp_stream.cu", "dp_stream_common.cuh", "dp_common.cuh"),
            workload="FSDP gradient reduce-scatter: K=8 virtual ranks x 64Mi bf16 N(0,1e-3), "
                     "ring-order fp32 fold, scale 1/8, fp32+bf16 shards",
            cfg={"K": K, "N_per_rank": N, "in_dtype": "bf16", "out_dtypes": ["f32", "bf16"],
                 "l2": "inputs 1 GiB per step > 129 MB L2; no flush"},
            e2e_in=bufs, e2e_out=o32 + o16, keep=(bufs, o32, o16))
    if name == "ar":
        K, N = K_RANKS, ar_mib * MiB // 4
        bufs = workloads.sweep_bufs_device(K, N, dev)
        return dict(
            step=lambda: B.dp_ring_allreduce(bufs, K, N, B.DP_FP32, 1.0 / K, sh),
            bytes=cm.all_reduce_hbm_bytes(K, N, "f32"), bound="hbm",
            kernel=("ar_vec_kernel<f32, K=8> (registers)" if variant == 1 else
                    "ar_tma_kernel<f32, K=8> (bulk copies through shared memory)"),
            traffic_key="ar_f32_k8" if variant == 1 else "ar_tma_f32_k8",
            src=(("dp_stream.cu", "dp_stream_common.cuh", "dp_common.cuh") if variant == 1
                 else ("dp_tma.cu", "dp_common.cuh")),
            workload=f"ring all-reduce in place: K=8 virtual ranks x {ar_mib} MiB fp32 U[-1,1], "
                     "ring-order fold, scale 1/8",
            cfg={"K": K, "N_per_rank": N, "dtype": "f32",
                 "l2": f"{2 * K * ar_mib} MiB per step > 129 MB L2; no flush"},
            e2e_in=bufs, e2e_out=bufs, keep=(bufs,))
    if name == "ag":
        K, C = K_RANKS, 32 * MiB // 4
        shards = [torch.randn(C, device=dev) for _ in range(K)]
        outs = [torch.empty(K * C, device=dev) for _ in range(K)]
        return dict(
            step=lambda: B.dp_all_gather(shards, K, C, B.DP_FP32, outs, sh),
            bytes=cm.all_gather_hbm_bytes(K, C, "f32"), bound="hbm",
            kernel=("ag_vec_kernel<K=8> (registers)" if variant == 1 else
                    "ag_tma_kernel (bulk copies through shared memory)"),
            traffic_key="ag_f32_k8" if variant == 1 else "ag_tma_f32_k8",
            src=(("dp_stream.cu", "dp_stream_common.cuh", "dp_common.cuh") if variant == 1
                 else ("dp_tma.cu", "dp_common.cuh")),
            workload="ring all-gather: K=8 shards of 32 MiB fp32 -> 8 x 256 MiB",
            cfg={"K": K, "shard_elems": C, "dtype": "f32",
                 "l2": "2.25 GiB per step > 129 MB L2; no flush"},
            e2e_in=shards, e2e_out=outs, keep=(shards, outs))
    if name in ("agmm_b", "agmm_a"):
        M, D, Kw, Fs = (8192, 4096, 8, 512) if name == "agmm_b" else (128, 512, 8, 64)
        g = torch.Generator(device=dev)
        g.manual_seed(40)
        x = (torch.randn(M, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        ws_ = [(torch.randn(Fs, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
               for _ in range(Kw)]
        y = torch.empty(M, Kw * Fs, dtype=torch.bfloat16, device=dev)
        # workspace for the chained split of a part-full last round (allocated once)
        wsb = B.dp_allgather_matmul_workspace_size(M, D, Kw, Fs)
        wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        return dict(
            step=lambda: B.dp_allgather_matmul(x, M, D, ws_, Kw, Fs, y, B.DP_BF16, sh,
                                               workspace=wsp, workspace_bytes=wsb),
            flops=cm.gemm_flops(M, Kw * Fs, D), bytes=cm.allgather_matmul_min_bytes(M, D, Kw * Fs),
            bound="tensor", kernel="agmm_kernel (tcgen05 kind::f16, TMA from 8 shards; a part-full "
                                   "last round split into chained segments through a workspace)",
            traffic_key=f"{name}", src=("dp_agmm.cu", "dp_common.cuh"),
            workload=f"FSDP all-gather fused into the local GEMM: x[{M},{D}] bf16, "
                     f"w_k[{Fs},{D}] x {Kw} -> y[{M},{Kw * Fs}] bf16, fp32 accumulate",
            cfg={"M": M, "D": D, "K": Kw, "F_shard": Fs, "y_dtype": "bf16",
                 "l2": "operands fit L2: a 512 MiB write flushes L2 before each timed launch"},
            e2e_in=[x] + ws_, e2e_out=[y], keep=(x, ws_, y, wsp), flush=True)
    if name in ("tp_ar", "tp_rs", "tp_fixture", "tp_rs_xw"):
        K = K_RANKS
        M, Ds, F = (1024, 64, 512) if name == "tp_fixture" else (8192, 512, 4096)
        xw = name == "tp_rs_xw"  # the x . w orientation: w_r [Ds, F]
        g = torch.Generator(device=dev)
        g.manual_seed(60)
        xs = [(torch.randn(M, Ds, generator=g, device=dev) * 0.02).to(torch.bfloat16)
              for _ in range(K)]
        ws_ = [(torch.randn(*((Ds, F) if xw else (F, Ds)), generator=g, device=dev) * 0.02)
               .to(torch.bfloat16) for _ in range(K)]
        scatter = name in ("tp_rs", "tp_rs_xw")
        rows = M // K if scatter else M
        ys = [torch.empty(rows, F, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        if xw:
            fn = B.dp_matmul_reduce_scatter_xw
        else:
            fn = B.dp_matmul_reduce_scatter if scatter else B.dp_matmul_allreduce
        out_bytes = K * rows * F * 2
        wsb = (B.dp_matmul_xw_workspace_size if xw else B.dp_matmul_workspace_size)(K, M, Ds, F)
        wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        return dict(
            step=lambda: fn(xs, ws_, K, M, Ds, F, ys, B.DP_BF16, 1.0, sh, workspace=wsp,
                            workspace_bytes=wsb),
            flops=cm.gemm_flops(M, F, K * Ds),
            bytes=K * (M * Ds + F * Ds) * 2 + out_bytes, bound="tensor",
            kernel="agmm_kernel (tcgen05, k-blocks of 8 ranks chained into one TMEM accumulator; "
                   "a part-full last round split into chained segments through a workspace)",
            traffic_key=name, src=("dp_agmm.cu", "dp_common.cuh"),
            workload=f"tensor-parallel psum fused into the GEMM: K=8 ranks x "
                     + (f"(x_r[{M},{Ds}] . w_r[{Ds},{F}]) summed, " if xw else
                        f"(x_r[{M},{Ds}] . w_r[{F},{Ds}]^T) summed, ")
                     + ("row shards [M/8, F] (reduce-scatter)" if scatter else
                        "[M, F] on every rank (all-reduce)") + ", bf16 out",
            cfg={"K": K, "M": M, "D_shard": Ds, "F": F, "mode": "rs" if scatter else "ar",
                 "w_layout": "[D_shard, F]" if xw else "[F, D_shard]",
                 "l2": "operands fit L2: a 512 MiB write flushes L2 before each timed launch"},
            e2e_in=xs + ws_, e2e_out=ys, keep=(xs, ws_, ys, wsp), flush=True)
    if name == "wgrad":
        # FSDP backward of the layer above (8192 tokens over K=8 ranks): the
        # weight gradient dW [4096, 4096] = sum_r dy_r^T x_r, reduce-scattered
        # in row shards [512, 4096]
        K, T, F, D = K_RANKS, 1024, 4096, 4096
        g = torch.Generator(device=dev)
        g.manual_seed(90)
        dys = [(torch.randn(T, F, generator=g, device=dev) * 0.02).to(torch.bfloat16)
               for _ in range(K)]
        xs = [(torch.randn(T, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
              for _ in range(K)]
        ys = [torch.empty(F // K, D, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        # workspace for the chained split of the last round (allocated once)
        wsb = B.dp_wgrad_workspace_size(K, T, F, D)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        return dict(
            step=lambda: B.dp_wgrad_reduce_scatter(dys, xs, K, T, F, D, ys, B.DP_BF16,
                                                   1.0 / K, sh, workspace=ws,
                                                   workspace_bytes=wsb),
            flops=cm.gemm_flops(F, D, K * T), bytes=K * T * (F + D) * 2 + F * D * 2,
            bound="tensor",
            kernel="agmm_kernel (tcgen05, MN-major operands, token blocks of 8 ranks chained "
                   "into one TMEM accumulator, row-shard epilogue; last round's tiles split "
                   "into chained segments through a workspace)",
            traffic_key=name, src=("dp_agmm.cu", "dp_common.cuh"),
            workload=f"FSDP backward weight gradient fused with its reduce-scatter: K=8 ranks x "
                     f"(dy_r[{T},{F}]^T . x_r[{T},{D}]) summed, row shards [{F // K}, {D}] bf16, "
                     f"scale 1/8",
            cfg={"K": K, "T_per_rank": T, "F": F, "D": D, "mode": "wgrad_rs",
                 "l2": "operands fit L2: a 512 MiB write flushes L2 before each timed launch"},
            e2e_in=dys + xs, e2e_out=ys, keep=(dys, xs, ys, ws), flush=True)
    if name.startswith("ddp"):
        # a GPT-2-small-shaped parameter list (124M parameters, 148 tensors),
        # fp32 gradients on K=8 ranks, bucketed all-reduce driven by the
        # Reducer with the parameters marked ready in backward (reverse) order
        from ring_allreduce_gradient_gb300.collectives import Reducer
        cap_mb = int(name[3:] or 25)
        K = K_RANKS
        numels = workloads.gpt2_small_numels()
        grads = workloads.ddp_grads_device(numels, K, dev)
        red = Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=cap_mb * MiB, scale=1.0 / K)
        ptrs = [[grads[r][p].data_ptr() for r in range(K)] for p in range(len(numels))]

        def eager():
            for p in reversed(range(len(numels))):
                red.mark_ready(p, ptrs[p], sh)
            st, _ = red.finish()
            assert st == B.DP_OK
        # One iteration captured in a CUDA graph: the replay is the device-side
        # cost of the bucket all-reduces (the eager, host-driven iteration pays
        # ~150 mark_ready calls of host time as well and is reported beside it).
        stream_obj = torch.cuda.ExternalStream(sh, device=dev)
        with torch.cuda.stream(stream_obj):
            eager()
            eager()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream_obj):
            eager()
        torch.cuda.synchronize()
        # the same iteration in the Reducer's overlap mode (DDP's asynchronous
        # all-reduce: buckets on two streams of the reducer's own, alternating,
        # joined to the caller's stream before the optimizer)
        red_o = Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=cap_mb * MiB, scale=1.0 / K)
        red_o.set_overlap(True)

        def eager_overlap():
            for p in reversed(range(len(numels))):
                red_o.mark_ready(p, ptrs[p], sh)
            st, _ = red_o.finish()
            assert st == B.DP_OK
            red_o.wait(sh)
        with torch.cuda.stream(stream_obj):
            eager_overlap()
            eager_overlap()
        torch.cuda.synchronize()
        graph_o = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_o, stream=stream_obj):
            eager_overlap()
        torch.cuda.synchronize()
        N = sum(numels)
        flat = [t for r in range(K) for t in grads[r]]
        def replay():
            with torch.cuda.stream(stream_obj):  # replay() launches on the current stream
                graph.replay()

        def replay_overlap():
            with torch.cuda.stream(stream_obj):
                graph_o.replay()

        return dict(
            step=replay, eager=eager, step_overlap=replay_overlap,
            bytes=cm.all_reduce_hbm_bytes(K, N, "f32"),
            bound="hbm", launches=red.num_buckets,
            kernel=("mt_ar_kernel<f32, K=8> (registers, one launch per bucket)" if variant == 1
                    else "mt_tma_kernel<f32, K=8> (bulk copies, one launch per bucket)"),
            traffic_key=name if variant != 1 else name + "_reg",
            src=("dp_bucket.cu", "dp_common.cuh") if variant == 1 else ("dp_tma.cu", "dp_common.cuh"),
            workload=f"DDP bucketed all-reduce: K=8 ranks x {len(numels)} fp32 gradient tensors "
                     f"({N} parameters, GPT-2-small shapes), bucket_cap {cap_mb} MiB -> "
                     f"{red.num_buckets} buckets, in place, ring order per bucket, scale 1/8; "
                     f"one Reducer iteration replayed from a CUDA graph",
            cfg={"K": K, "params": N, "tensors": len(numels), "bucket_cap_mib": cap_mb,
                 "buckets": red.num_buckets, "l2": "4 GB per step > 129 MB L2; no flush"},
            e2e_in=flat, e2e_out=flat, keep=(grads, red, graph, red_o, graph_o))
    if name == "odc":
        K, N, L = K_RANKS, 16 * MiB, odc_layers
        m, toks = workloads.odc_schedule(K)
        Mx = max(m)
        grads = [[[workloads.odc_grad(l, r, j, N, int(toks[r, j]), dev) for j in range(m[r])]
                  for r in range(K)] for l in range(L)]
        tables = [[gg for r in range(K) for gg in (grads[l][r] + [None] * (Mx - m[r]))]
                  for l in range(L)]
        o32 = [torch.empty(N // K, device=dev) for _ in range(K)]
        o16 = [torch.empty(N // K, dtype=torch.bfloat16, device=dev) for _ in range(K)]

        def step():
            for l in range(L):
                B.dp_odc_reduce_scatter(tables[l], m, K, Mx, N, B.DP_BF16, o32, o16, 1.0 / K,
                                        sh)
        flat = [gg for l in range(L) for r in range(K) for gg in grads[l][r]]
        return dict(
            step=step, launches=L,
            bytes=L * cm.odc_fused_hbm_bytes(sum(m), N, "bf16", ("f32", "bf16")), bound="hbm",
            kernel="odc_vec_kernel<bf16, fp32+bf16 out>", traffic_key="odc_fused_bf16_k8",
            src=("dp_odc.cu", "dp_stream_common.cuh", "dp_common.cuh"),
            workload=f"variable-length step, unpadded: K=8 ranks, {L} layers x 16Mi bf16, "
                     f"microbatches per rank {m}, fused accumulate + ring reduce-scatter",
            cfg={"K": K, "N_per_layer": N, "layers": L, "microbatches": m,
                 "l2": "1.2 GiB per layer > 129 MB L2; no flush"},
            e2e_in=flat, e2e_out=o32 + o16, keep=(grads, tables, o32, o16))
    raise ValueError(name)

# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    from ring_allreduce_gradient_gb300 import binding as B
    from ring_allreduce_gradient_gb300 import build as cuda_build

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
    B.dp_set_collective_variant(args.variant)
    hbm_peak, bf16_peak, bf16_sus, peak_kind = peaks()

    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    wl = make_workload(args.workload, dev, sh, args.odc_layers, args.ar_mib)
    step = wl["step"]
    tensor_bound = wl["bound"] == "tensor"
    work = wl["flops"] if tensor_bound else wl["bytes"]
    scale_unit = 1e12 if tensor_bound else 1e9
    unit = "TFLOP/s" if tensor_bound else "GB/s"
    launches_per_step = wl.get("launches", 1)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    # ---- timed region ----
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    flush = torch.empty(512 * MiB // 4, device=dev) if wl.get("flush") else None
    with ClockSampler(local) as clk:
        start.record(stream)
        for i, (a, b) in enumerate(per):
            if flush is not None:  # evict the L2-resident operands (outside the step's events)
                with torch.cuda.stream(stream):
                    flush.fill_(float(i))
            a.record(stream)
            step()
            b.record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in per]
    # with flushes in between, the job time is the steps' own time
    elapsed_ms = sum(step_ms) if flush is not None else start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    st = B.dp_get_device_error(sh)
    assert st == B.DP_OK, B.status_string(st)

    value = aggregate_rate(work, args.steps, ws, elapsed_ms, scale_unit)
    avg_launch_ms = statistics.mean(step_ms) / launches_per_step
    median_launch_ms = statistics.median(step_ms) / launches_per_step
    achieved = (work / launches_per_step) / (avg_launch_ms * 1e-3) / scale_unit
    peak = bf16_peak if tensor_bound else hbm_peak
    src_hash = source_hash(*wl["src"])
    desc, cfg, kern, tkey = wl["workload"], wl["cfg"], wl["kernel"], wl["traffic_key"]

    # ---- end to end: pinned host inputs -> device -> the same call -> host ----
    e2e = None
    if not args.no_e2e:
        hin = [torch.empty_like(t, device="cpu").pin_memory() for t in wl["e2e_in"]]
        for h, t in zip(hin, wl["e2e_in"]):
            h.copy_(t)
        hout = [torch.empty_like(t, device="cpu").pin_memory() for t in wl["e2e_out"]]

        def e2e_step():
            with torch.cuda.stream(stream):
                for t, h in zip(wl["e2e_in"], hin):
                    t.copy_(h, non_blocking=True)
                step()
                for h, t in zip(hout, wl["e2e_out"]):
                    h.copy_(t, non_blocking=True)

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
        e2e_ms = max_over_ranks(a.elapsed_time(b), dev)
        e2e = {"value": round(aggregate_rate(work, e2e_steps, ws, e2e_ms, scale_unit), 3),
               "unit": unit,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in wl["e2e_in"]),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in wl["e2e_out"]),
               "ms_per_step": e2e_ms / e2e_steps}
        del hin, hout

    if e2e is not None and args.workload == "rs":
        pe = e2e_pipelined_rs(wl, dev, stream, min(max(args.steps, 4), 20))
        pe_ms = max_over_ranks(pe["ms_per_step"], dev)
        zc_ms = max_over_ranks(pe["zero_copy_ms_per_step"], dev)
        e2e.update({
            "mode": "pipelined: step i's H2D overlaps step i-1's kernel and D2H (double "
                    "buffers, three streams); median of three runs",
            "pipelined_runs_ms_per_step": pe["runs_ms_per_step"],
            "value": round(aggregate_rate(work, 1, ws, pe_ms, scale_unit), 3),
            "ms_per_step": pe_ms,
            "sequential_value": e2e["value"], "sequential_ms_per_step": e2e["ms_per_step"],
            "zero_copy_value": round(aggregate_rate(work, 1, ws, zc_ms, scale_unit), 3),
            "zero_copy_ms_per_step": zc_ms,
            "zero_copy_note": "the kernel reads pinned host inputs and writes pinned host "
                              "shards directly over NVLink-C2C (no copy calls)"})

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and args.workload == "rs":
        cpu = cpu_baseline_rs(wl["e2e_in"], args.cpu_sample_mib)

    rows = None
    if ws == 1 and not args.no_rows and args.workload == "rs":
        del wl, step
        torch.cuda.empty_cache()
        try:
            rows = measure_rows(dev, stream, hbm_peak, bf16_peak, peak_kind, args)
            if not args.no_cpu_baseline:
                rows["cpu_oracle"] = cpu_oracle_rows()
        except Exception as exc:  # the headline line is still printed
            import traceback
            traceback.print_exc()
            rows = {"error": f"{type(exc).__name__}: {exc}"}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": unit,
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": dict(workload=desc, **cfg,
                           parallelism=f"replicas x{ws} (K virtual ranks on each GPU)"),
            "roofline": {
                "kernel": kern,
                "bound": "tensor" if tensor_bound else "hbm",
                "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": f"{peak_kind}, burst ("
                             + ("cuBLAS bf16 dense" if tensor_bound else "copy bandwidth") + ")",
                "unit": unit, "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic(tkey, src_hash),
                "algorithmic_per_launch": work / launches_per_step,
                "avg_launch_ms": avg_launch_ms,
                "median_launch_ms": median_launch_ms,
                "max_launch_ms": max(step_ms) / launches_per_step,
            },
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clk.summary(),
            "rows": rows,
        }
        if rows is not None:
            line["summary"] = rows_summary(rows, cpu)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def e2e_pipelined_rs(wl, dev, stream, steps):
    """End-to-end headline step with host buffers: every step copies its K
    inputs from pinned host memory, runs the reduce-scatter and copies both
    shard sets back; the copies of consecutive steps overlap (H2D of step i
    with the kernel and D2H of step i-1) through double buffers on three
    streams.  Also times the same call on the pinned host buffers directly
    (zero-copy).  Returns per-step milliseconds."""
    import torch

    from ring_allreduce_gradient_gb300 import binding as B

    K, N = K_RANKS, N_ELEMS
    C = N // K
    bufs, o32, o16 = wl["keep"]
    sets = [(bufs, o32, o16),
            ([torch.empty_like(b) for b in bufs], [torch.empty_like(t) for t in o32],
             [torch.empty_like(t) for t in o16])]
    hin = [torch.empty_like(b, device="cpu").pin_memory() for b in bufs]
    for h, b in zip(hin, bufs):
        h.copy_(b)
    hout = [([torch.empty_like(t, device="cpu").pin_memory() for t in o32],
             [torch.empty_like(t, device="cpu").pin_memory() for t in o16]) for _ in range(2)]
    s_h2d = torch.cuda.Stream(device=dev)
    s_d2h = torch.cuda.Stream(device=dev)
    comp = stream
    ev = lambda: torch.cuda.Event()
    comp_done = [None, None]
    d2h_done = [None, None]

    def step(i):
        k = i % 2
        bk, k32, k16 = sets[k]
        if comp_done[k] is not None:
            s_h2d.wait_event(comp_done[k])  # the kernel of step i-2 is done with set k
        with torch.cuda.stream(s_h2d):
            for b, h in zip(bk, hin):
                b.copy_(h, non_blocking=True)
        e_in = ev()
        e_in.record(s_h2d)
        comp.wait_event(e_in)
        if d2h_done[k] is not None:
            comp.wait_event(d2h_done[k])  # set k's shards of step i-2 are read out
        B.dp_reduce_scatter_dual(bk, K, N, B.DP_BF16, k32, k16, 1.0 / K, comp.cuda_stream)
        e_c = ev()
        e_c.record(comp)
        comp_done[k] = e_c
        s_d2h.wait_event(e_c)
        with torch.cuda.stream(s_d2h):
            for h, t in zip(hout[k][0], k32):
                h.copy_(t, non_blocking=True)
            for h, t in zip(hout[k][1], k16):
                h.copy_(t, non_blocking=True)
        e_o = ev()
        e_o.record(s_d2h)
        d2h_done[k] = e_o

    def timed(fn, n):
        main = torch.cuda.current_stream(dev)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for st_ in (s_h2d, comp, s_d2h):
            st_.wait_event(a)
        for i in range(n):
            fn(i)
        for st_ in (s_h2d, comp, s_d2h):
            e = ev()
            e.record(st_)
            main.wait_event(e)
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    for i in range(2):
        step(i)
    # three runs, the median reported: the host link is shared with the rest
    # of the machine, and one slow run should not set the number
    runs = [timed(step, steps) for _ in range(3)]
    pipelined = statistics.median(runs)
    h32, h16 = hout[0]
    zc = lambda i: B.dp_reduce_scatter_dual(hin, K, N, B.DP_BF16, h32, h16, 1.0 / K,
                                            comp.cuda_stream)
    zc(0)
    zero_copy = timed(zc, steps)
    del sets, hin, hout
    return {"ms_per_step": pipelined, "zero_copy_ms_per_step": zero_copy,
            "runs_ms_per_step": [round(r, 4) for r in runs]}


def cpu_baseline_rs(bufs, sample_mib, min_seconds=10.0, max_reps=30):
    """The oracle's ring simulator on the first sample_mib Mi elements of every
    rank's gradient (the same data), single-threaded on the host, repeated
    until about min_seconds of CPU work."""
    import oracle
    import workloads
    from ring_allreduce_gradient_gb300 import costmodel as cm

    K = len(bufs)
    n = min(sample_mib * MiB, bufs[0].numel())
    n -= n % K
    host = [workloads.torch_bf16_to_bits(b[:n]) for b in bufs]
    reps, t_total = 0, 0.0
    while reps < max_reps and (reps == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        oracle.reduce_scatter(host, 1.0 / K)
        t_total += time.perf_counter() - t0
        reps += 1
    nbytes = cm.reduce_scatter_hbm_bytes(K, n, "bf16", ("f32", "bf16"))
    # the same simulator on element slabs across every core this process may use
    cores = len(os.sched_getaffinity(0))
    treps, t_thr = 0, 0.0
    while treps < max_reps and (treps == 0 or t_thr < min_seconds / 3):
        t0 = time.perf_counter()
        oracle.reduce_scatter_threaded(host, 1.0 / K, threads=cores)
        t_thr += time.perf_counter() - t0
        treps += 1
    return {"value": round(nbytes * reps / t_total / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "seconds": round(t_total, 3),
            "sample": f"ring step simulator, K={K} ranks x {n} bf16 elements "
                      f"({n / bufs[0].numel():.3f} of each rank's 64Mi gradient, the same "
                      f"data), {reps} call(s)",
            "threaded": {"value": round(nbytes * treps / t_thr / 1e9, 4), "unit": "GB/s",
                         "cores": cores, "seconds": round(t_thr, 3),
                         "sample": f"the same simulator on {cores} element slabs at once "
                                   f"(one thread each), same data, {treps} call(s)"}}


def cpu_oracle_rows(budget_s=2.0):
    """The oracle, as it stands, on bounded samples of the other configs'
    workloads (single-threaded, on the host cores), each repeated to about
    `budget_s` seconds: the parity all-reduce (K=4 x 4096 integer fp32), the
    all-reduce sweep's K=8 x 1 MiB point, the 4(a) GEMM in fp64 (the whole
    x[128,512] . w[512,512]^T), 4096 sampled outputs of the 4(b) GEMM, and
    one variable-length layer on a 256 Ki sample of every microbatch
    gradient.  A reported baseline only."""
    import numpy as np
    import oracle
    import workloads
    from ring_allreduce_gradient_gb300 import costmodel as cm

    def rate(fn):
        reps, t = 0, 0.0
        while reps == 0 or (t < budget_s and reps < 1000):
            t0 = time.perf_counter()
            fn()
            t += time.perf_counter() - t0
            reps += 1
        return t / reps

    out = {}
    bufs = workloads.ring_ints(K=4, N=4096, seed=0)
    dt = rate(lambda: oracle.all_reduce(bufs, 1.0))
    out["allreduce_k4_4096_ints_us"] = round(dt * 1e6, 1)
    N = 1 << 18  # 1 MiB of fp32 per rank
    sb = workloads.sweep_bufs(8, N)
    dt = rate(lambda: oracle.all_reduce(sb, 1.0 / 8))
    out["allreduce_k8_1MiB_GBps"] = round(cm.all_reduce_hbm_bytes(8, N, "f32") / dt / 1e9, 3)
    x, ws = workloads.gemm_operands(128, 512, 8, 64)
    dt = rate(lambda: oracle.allgather_matmul_f64(x, ws))
    out["gemm_4a_f64_GFLOPs"] = round(2 * 128 * 512 * 512 / dt / 1e9, 3)
    # 4(b) whole would take minutes in fp64: 4096 sampled outputs of it
    x4, ws4 = workloads.gemm_operands(8192, 4096, 8, 512)
    rs = np.random.default_rng(11)
    ms, fs = rs.integers(0, 8192, 4096), rs.integers(0, 4096, 4096)
    dt = rate(lambda: oracle.allgather_matmul_f64_sampled(x4, ws4, ms, fs))
    out["gemm_4b_f64_sampled_GFLOPs"] = round(2 * 4096 * ms.size / dt / 1e9, 3)
    del x4, ws4
    m, toks = workloads.odc_schedule(8)
    n = 1 << 18
    rng = np.random.default_rng(9)
    grads = [[workloads.to_bf16_bits(rng.standard_normal(n).astype(np.float32) *
                                     np.float32(1e-3 * toks[r, j])) for j in range(m[r])]
             for r in range(8)]
    dt = rate(lambda: oracle.odc_layer(grads, m, 1.0 / 8, n))
    out["odc_layer_GBps"] = round(cm.odc_fused_hbm_bytes(sum(m), n, "bf16", ("f32", "bf16")) /
                                  dt / 1e9, 3)
    out["sample"] = ("single-threaded oracle; the sweep point, the 4(a) GEMM, 4096 sampled "
                     "outputs of the 4(b) GEMM and a 256 Ki-element sample of one "
                     "variable-length layer (microbatches " + str(m) + ")")
    return out


# ----------------------------------------------------------------------------
# the other rows, measured at N=1 after the headline
# ----------------------------------------------------------------------------

def measure_rows(dev, stream, hbm_peak, bf16_peak, peak_kind, args):
    """Median device time of each other row's step (CUDA events on `stream`)."""
    import torch

    from ring_allreduce_gradient_gb300 import binding as B
    from ring_allreduce_gradient_gb300 import costmodel as cm

    sh = stream.cuda_stream
    rows = {}
    reps = args.row_reps

    mins = {}
    flush_buf = torch.empty(512 * MiB // 4, device=dev)
    clean_buf = torch.ones(512 * MiB // 4, device=dev)

    def timed(fn, n, key=None, flush=False, clean=False):
        # at least 6 warm-up calls, then the median of n timed ones (the
        # minimum is kept beside it); with `flush`, a 512 MiB write between
        # timed calls evicts the operands from L2 (for working sets that fit);
        # with `clean` as well, a 512 MiB read of another buffer then leaves
        # L2 holding clean lines instead of the write's dirty ones
        with torch.cuda.stream(stream):
            for _ in range(6):
                fn()
            if not flush:
                ts = time_events(fn, n, stream)
            else:
                evs = []
                for i in range(n):
                    flush_buf.fill_(float(i))
                    if clean:
                        clean_buf.sum()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
                        enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    evs.append((a, b))
                torch.cuda.synchronize()
                ts = [a.elapsed_time(b) for a, b in evs]
        if key is not None:
            mins[key] = min(ts)
        return statistics.median(ts)

    def graph_launch_us(fn, per_graph=20, replays=10):
        # latency-bound rows: the per-launch device time with the host out of
        # the way, `per_graph` launches captured in one CUDA graph and replayed
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per_graph):
                fn()
        with torch.cuda.stream(stream):
            g.replay()
            ts = time_events(g.replay, replays, stream)
        del g
        return round(statistics.median(ts) * 1e3 / per_graph, 2)

    names = [("ar", 1), ("ar", 2), ("ag", 1), ("ag", 2), ("agmm_b", 0), ("agmm_a", 0),
             ("tp_ar", 0), ("tp_rs", 0), ("tp_rs_xw", 0), ("tp_fixture", 0), ("wgrad", 0),
             ("ddp1", 0), ("ddp25", 0), ("ddp100", 0)]
    for name, variant in names:
        prev = B.dp_get_collective_variant()
        if variant:
            B.dp_set_collective_variant(variant)
        wl = make_workload(name, dev, sh)
        try:
            ms = timed(wl["step"], reps, "row", flush=wl.get("flush", False))
        finally:
            B.dp_set_collective_variant(prev)
        if variant:
            name = f"{name}_{'registers' if variant == 1 else 'bulk_copy'}"
        r = {"workload": wl["workload"], "ms": ms, "min_ms": mins["row"]}
        if name in ("agmm_a", "tp_fixture"):
            r["graph_us"] = graph_launch_us(wl["step"])
        if "step_overlap" in wl:
            oms = timed(wl["step_overlap"], reps)
            r["overlap_mode_ms"] = oms
            r["overlap_mode_GB/s"] = round(wl["bytes"] / (oms * 1e-3) / 1e9, 1)
            r["overlap_mode_frac_hbm"] = round(wl["bytes"] / (oms * 1e-3) / 1e9 / hbm_peak, 4)
        if "eager" in wl:
            ems = timed(wl["eager"], max(3, reps // 2))
            r["eager_ms"] = ems
            r["eager_GB/s"] = round(wl["bytes"] / (ems * 1e-3) / 1e9, 1)
        if wl["bound"] == "tensor":
            tf = wl["flops"] / (ms * 1e-3) / 1e12
            r.update({"TFLOP/s": round(tf, 1), "frac_bf16": round(tf / bf16_peak, 4),
                      "peak": f"{bf16_peak} TFLOP/s ({peak_kind}, burst)"})
            if wl.get("flush"):  # the same launches back to back, operands warm in L2
                wms = timed(wl["step"], reps)
                wtf = wl["flops"] / (wms * 1e-3) / 1e12
                cms = timed(wl["step"], reps, flush=True, clean=True)
                ctf = wl["flops"] / (cms * 1e-3) / 1e12
                r.update({"l2": "flushed before each timed launch", "warm_ms": wms,
                          "warm_TFLOP/s": round(wtf, 1),
                          "warm_frac_bf16": round(wtf / bf16_peak, 4),
                          "clean_l2_ms": cms, "clean_l2_TFLOP/s": round(ctf, 1),
                          "clean_l2_frac_bf16": round(ctf / bf16_peak, 4)})
        else:
            gbs = wl["bytes"] / (ms * 1e-3) / 1e9
            r.update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4)})
        rows[name] = r
        st = B.dp_get_device_error(sh)
        assert st == B.DP_OK, B.status_string(st)
        del wl
        torch.cuda.empty_cache()

    # the 4(b) GEMM once more as a sustained run (about half a second of
    # back-to-back launches) with the SM clocks sampled meanwhile, against
    # the sustained bf16 peak
    wl = make_workload("agmm_b", dev, sh)
    with torch.cuda.stream(stream):
        for _ in range(20):
            wl["step"]()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            ts = time_events(wl["step"], 3000, stream)
    ms = statistics.median(ts)
    tf = wl["flops"] / (ms * 1e-3) / 1e12
    sus = peaks()[2]
    rows["agmm_b_sustained"] = {"launches": len(ts), "ms": ms, "TFLOP/s": round(tf, 1),
                                "frac_bf16_sustained": round(tf / sus, 4),
                                "peak": f"{sus} TFLOP/s (measured, sustained)",
                                "clocks": clk.summary()}
    del wl
    torch.cuda.empty_cache()

    # variable-length step: fused unpadded / padded, and the two-phase path
    # (one accumulate launch per microbatch, padding buckets included, then
    # the reduce-scatter of the fp32 accumulators)
    wl = make_workload("odc", dev, sh, args.odc_layers)
    grads, tables, o32, o16 = wl["keep"]
    K, N, L = K_RANKS, 16 * MiB, args.odc_layers
    m = wl["cfg"]["microbatches"]
    Mx = max(m)
    accs = [torch.empty(N, device=dev) for _ in range(K)]

    def fused(pad):
        mm = [Mx] * K if pad else m
        for l in range(L):
            B.dp_odc_reduce_scatter(tables[l], mm, K, Mx, N, B.DP_BF16, o32, o16, 1.0 / K, sh)

    def two_phase(pad):
        for l in range(L):
            for r in range(K):
                for j in range(Mx if pad else m[r]):
                    g = grads[l][r][j] if j < m[r] else None
                    B.dp_grad_accumulate(accs[r], g, N, B.DP_BF16, j == 0, sh)
            B.dp_reduce_scatter_dual(accs, K, N, B.DP_FP32, o32, o16, 1.0 / K, sh)

    res = {"workload": wl["workload"]}
    n = max(3, reps // 4)
    for key, fn in (("fused_nopad", lambda: fused(False)), ("fused_pad", lambda: fused(True)),
                    ("two_phase_nopad", lambda: two_phase(False)),
                    ("two_phase_pad", lambda: two_phase(True))):
        res[key] = {"ms_per_step": timed(fn, n)}
    gbs = wl["bytes"] / (res["fused_nopad"]["ms_per_step"] * 1e-3) / 1e9
    res["fused_nopad"].update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4)})
    tp_bytes = 0
    for r in range(K):
        tp_bytes += cm.accumulate_hbm_bytes(N, "bf16", True)
        tp_bytes += (m[r] - 1) * cm.accumulate_hbm_bytes(N, "bf16", False)
    tp_bytes = L * (tp_bytes + cm.reduce_scatter_hbm_bytes(K, N, "f32", ("f32", "bf16")))
    gbs = tp_bytes / (res["two_phase_nopad"]["ms_per_step"] * 1e-3) / 1e9
    res["two_phase_nopad"].update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4)})
    res["pad_over_nopad_fused"] = round(res["fused_pad"]["ms_per_step"] /
                                        res["fused_nopad"]["ms_per_step"], 4)
    res["pad_over_nopad_two_phase"] = round(res["two_phase_pad"]["ms_per_step"] /
                                            res["two_phase_nopad"]["ms_per_step"], 4)
    rows["odc"] = res
    rows["settle_pipeline"] = measure_settle_pipeline(dev, grads, m, L, N, max(3, reps // 4))
    rows["ddp_overlap"] = measure_ddp_overlap(dev, max(3, reps // 4))
    rows["c3"] = measure_c3(dev)
    rows["allreduce_sweep"] = measure_sweep(dev, hbm_peak)
    st = B.dp_get_device_error(sh)
    assert st == B.DP_OK, B.status_string(st)
    del wl, grads, tables, accs, o32, o16
    torch.cuda.empty_cache()
    return rows


def rows_summary(rows, cpu):
    """The rows' key figures in about a kilobyte, printed as the last key of
    the line so that a reader keeping only the end of the output still has
    every row; the most important last (fractions are of the measured
    peaks; "warm" = the same launches back to back, operands in L2)."""
    if not rows or "error" in rows:
        return {"rows": (rows or {}).get("error", "not measured")}
    out = {}
    if cpu and "threaded" in cpu:
        out["cpu_oracle_GBps"] = [cpu["value"], cpu["threaded"]["value"],
                                  f'{cpu["threaded"]["cores"]} cores']
    co = rows.get("cpu_oracle")
    if co:
        out["cpu_oracle_rows"] = {k: v for k, v in co.items() if k != "sample"}
    sw = rows.get("allreduce_sweep")
    if sw:
        fr = {}
        for v in sw.values():
            if v.get("bytes_per_rank", 0) >= 64 * MiB:
                fr.setdefault(f"K{v['K']}", []).append(round(v.get("allreduce_frac", 0), 3))
        out["ar_frac_64M_256M_1G"] = fr
        out["ar_frac_64M_clean_l2"] = {f"K{v['K']}": round(v.get("allreduce_frac_clean_l2", 0), 3)
                                       for v in sw.values() if v.get("bytes_per_rank") == 64 * MiB}
    c3 = rows.get("c3")
    if c3:
        out["c3_best_S"] = {c: max((v.get("S", 0) for v in var.values()), default=None)
                            for c, var in c3.items() if isinstance(var, dict)}
    for key in ("ddp_overlap", "settle_pipeline"):
        r = rows.get(key)
        r = r.get("best", r) if key == "settle_pipeline" and r else r
        if r and "S" in r:
            out[key] = {"S": r["S"], "pct_ideal": r["pct_of_ideal"]}
    o = rows.get("odc")
    if o and "fused_nopad" in o:
        out["odc"] = {"frac": o["fused_nopad"].get("frac_hbm"),
                      "pad/nopad": o.get("pad_over_nopad_fused")}
    for name in ("ddp1", "ddp25", "ddp100", "ag_bulk_copy", "ar_bulk_copy"):
        r = rows.get(name)
        if r and "frac_hbm" in r:
            out[name.replace("_bulk_copy", "") + "_frac"] = r["frac_hbm"]
        if r and "overlap_mode_frac_hbm" in r:
            out[name + "_overlap_mode_frac"] = r["overlap_mode_frac_hbm"]
    for name in ("tp_fixture", "agmm_a"):
        r = rows.get(name)
        if r:
            out[name + "_us"] = round(r["ms"] * 1e3, 2)
            if "graph_us" in r:
                out[name + "_graph_us"] = r["graph_us"]
    for name in ("tp_ar", "tp_rs_xw", "tp_rs", "wgrad"):
        r = rows.get(name)
        if r and "frac_bf16" in r:
            out[name] = {"frac": r["frac_bf16"], "warm": r.get("warm_frac_bf16")}
    r = rows.get("agmm_b_sustained")
    if r:
        c = r.get("clocks", {})
        out["agmm_b_sustained"] = {"TFLOP/s": r["TFLOP/s"], "frac": r["frac_bf16_sustained"],
                                   "sm_mhz": c.get("sm_mhz"), "reasons": c.get("reasons")}
    r = rows.get("agmm_b")
    if r and "TFLOP/s" in r:
        out["agmm_b"] = {"TFLOP/s": r["TFLOP/s"], "frac": r["frac_bf16"],
                         "clean_l2_frac": r.get("clean_l2_frac_bf16"),
                         "warm_TFLOP/s": r.get("warm_TFLOP/s"),
                         "warm_frac": r.get("warm_frac_bf16"), "us": round(r["ms"] * 1e3, 1)}
    return out


# ----------------------------------------------------------------------------
# the all-reduce bandwidth sweep (K in {2,4,8}, 4 KiB .. 1 GiB per rank)
# ----------------------------------------------------------------------------

def measure_sweep(dev, hbm_peak, reps=10):
    """Fused in-place all-reduce and the composed reduce-scatter + all-gather
    over the sweep's per-rank sizes.  Where the K buffers fit in L2 the
    cache is flushed (a 512 MiB write) before every timed call, so the
    numbers are HBM numbers; the median of `reps` calls is reported with the
    algorithmic bytes (read K*N*4 + write K*N*4 for the all-reduce).  The
    write leaves L2 full of dirty lines that the timed call then writes back;
    the all-reduce is also timed after the write plus a 512 MiB read of
    another buffer (`*_clean_l2`: inputs still evicted, L2 holding clean
    lines)."""
    import torch

    from ring_allreduce_gradient_gb300 import binding as B
    from ring_allreduce_gradient_gb300 import costmodel as cm
    import workloads

    st = torch.cuda.Stream(device=dev)
    sh = st.cuda_stream
    flush = torch.empty(512 * MiB // 4, device=dev)
    clean = torch.ones(512 * MiB // 4, device=dev)
    out = {}
    for K in (2, 4, 8):
        for nbytes in workloads.sweep_sizes_bytes():
            N = nbytes // 4
            bufs = workloads.sweep_bufs_device(K, N, dev)
            C = N // K
            shards = [torch.empty(C, device=dev) for _ in range(K)]
            outs = [torch.empty(N, device=dev) for _ in range(K)]
            cold = K * nbytes * 2 <= 256 * MiB

            def timed(fn, clean_l2=False):
                ts = []
                with torch.cuda.stream(st):
                    for i in range(reps + 2):
                        if cold or clean_l2:
                            flush.fill_(float(i))
                        if clean_l2:  # read another 512 MiB: L2 left holding clean lines
                            clean.sum()
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
                            enable_timing=True)
                        a.record(st)
                        fn()
                        b.record(st)
                        if i >= 2:
                            ts.append((a, b))
                torch.cuda.synchronize()
                return statistics.median(a.elapsed_time(b) for a, b in ts)

            t_ar = timed(lambda: B.dp_ring_allreduce(bufs, K, N, B.DP_FP32, 1.0 / K, sh))
            t_ar_clean = timed(lambda: B.dp_ring_allreduce(bufs, K, N, B.DP_FP32, 1.0 / K, sh),
                               clean_l2=True)
            prev = B.dp_get_collective_variant()
            try:
                B.dp_set_collective_variant(1)
                t_ar_reg = timed(lambda: B.dp_ring_allreduce(bufs, K, N, B.DP_FP32, 1.0 / K, sh))
                B.dp_set_collective_variant(2)
                t_ar_bulk = timed(lambda: B.dp_ring_allreduce(bufs, K, N, B.DP_FP32, 1.0 / K, sh))
            finally:
                B.dp_set_collective_variant(prev)
            t_rsag = timed(lambda: (B.dp_reduce_scatter(bufs, K, N, B.DP_FP32, shards, 1.0 / K,
                                                        B.DP_FP32, sh),
                                    B.dp_all_gather(shards, K, C, B.DP_FP32, outs, sh)))
            ar_bytes = cm.all_reduce_hbm_bytes(K, N, "f32")
            rsag_bytes = (cm.reduce_scatter_hbm_bytes(K, N, "f32", ("f32",)) +
                          cm.all_gather_hbm_bytes(K, C, "f32"))
            g_ar = ar_bytes / (t_ar * 1e-3) / 1e9
            g_rsag = rsag_bytes / (t_rsag * 1e-3) / 1e9
            out[f"K{K}_{nbytes}B"] = {
                "K": K, "bytes_per_rank": nbytes, "cold_l2": cold,
                "allreduce_us": round(t_ar * 1e3, 2), "allreduce_GBps": round(g_ar, 1),
                "allreduce_frac": round(g_ar / hbm_peak, 4),
                "allreduce_us_clean_l2": round(t_ar_clean * 1e3, 2),
                "allreduce_frac_clean_l2": round(ar_bytes / (t_ar_clean * 1e-3) / 1e9 / hbm_peak, 4),
                "allreduce_us_registers": round(t_ar_reg * 1e3, 2),
                "allreduce_us_bulk_copy": round(t_ar_bulk * 1e3, 2),
                "rs_ag_us": round(t_rsag * 1e3, 2), "rs_ag_GBps": round(g_rsag, 1),
                "ring_transport_bytes_per_rank": cm.ring_allreduce_bytes_per_rank(nbytes, K)}
            del bufs, shards, outs
        torch.cuda.empty_cache()
    st_ = B.dp_get_device_error(sh)
    assert st_ == B.DP_OK, B.status_string(st_)
    return out


# ----------------------------------------------------------------------------
# the cross-iteration settle pipeline
# ----------------------------------------------------------------------------

def measure_settle_pipeline(dev, grads, m, L, N, reps):
    """The settle pipeline of "Using ODC to Accelerate AMD SFT Training",
    "Discussion: Settle Does Not Yet Overlap with Backward", on the
    variable-length workload: the minibatch's microbatches in two groups
    (j < 4, j >= 4), every group's backward stood in for by one 4(b) GEMM per
    layer (x[8192,4096] . w^T, 0.16 ms), every (group, layer) settled by
    dp_odc_settle_group / the pipe.  Schedules: serial (GEMMs and settles in
    order on one stream), per_group (the page's: after a group's backward,
    its L settles are pushed and run beside the next group's backward; one
    join), per_layer (each layer's settle pushed right after its GEMM).
    S = T_serial / T_schedule with T_serial the serial schedule at full
    speed, S_ideal = T_serial / max(T_gemms, T_settles), % of ideal =
    (S - 1) / (S_ideal - 1) ("Optimizing ML Concurrent Computation and
    Communication with GPU DMA Engines", Problem Formulation).  Variants cap
    the pipe's settle CTAs (and the GEMM's, partitioned)."""
    import torch

    from ring_allreduce_gradient_gb300 import binding as B

    K = K_RANKS
    bounds = [0, 4, max(max(m), 4)]
    G = len(bounds) - 1
    C = N // K
    accs = [[torch.empty(C, device=dev) for _ in range(K)] for _ in range(L)]
    o32 = [torch.empty(C, device=dev) for _ in range(K)]
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    tables = []
    for g in range(G):
        lo, hi = bounds[g], bounds[g + 1]
        cnt = [max(0, min(hi, m[r]) - lo) for r in range(K)]
        gm = max(cnt)
        per_layer = []
        for l in range(L):
            t = []
            for r in range(K):
                row = grads[l][r][lo:lo + cnt[r]]
                t.extend(row + [None] * (gm - len(row)))
            per_layer.append(t)
        tables.append((per_layer, cnt, gm))
    wl = make_workload("agmm_b", dev, 0)
    sa = torch.cuda.Stream(device=dev)
    sh = sa.cuda_stream
    # the GEMM workload's closure launches on stream 0; rebuild it on sa
    x, ws_, y, wsp = wl["keep"]
    wsb = B.dp_allgather_matmul_workspace_size(8192, 4096, 8, 512)

    def gemm():
        B.dp_allgather_matmul(x, 8192, 4096, ws_, 8, 512, y, B.DP_BF16, sh, workspace=wsp,
                              workspace_bytes=wsb)

    def phase(g):
        return (B.DP_SETTLE_FIRST if g == 0 else 0) | (B.DP_SETTLE_LAST if g == G - 1 else 0)

    def settle_direct(g, l):
        t, cnt, gm = tables[g]
        B.dp_odc_settle_group(t[l], cnt, K, gm, N, B.DP_BF16, accs[l], phase(g), o32, o16,
                              1.0 / K, sh)

    def timed(fn):
        ts = []
        for i in range(reps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(sa)
            fn()
            b.record(sa)
            torch.cuda.synchronize()
            if i >= 2:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def gemms_only():
        for _ in range(G * L):
            gemm()

    def settles_only():
        for g in range(G):
            for l in range(L):
                settle_direct(g, l)

    def serial():
        for g in range(G):
            for l in range(L):
                gemm()
            for l in range(L):
                settle_direct(g, l)

    t_gemm, t_settle, t_serial = timed(gemms_only), timed(settles_only), timed(serial)
    s_ideal = t_serial / max(t_gemm, t_settle)
    out = {"groups": bounds, "layers": L, "T_gemms_ms": round(t_gemm, 3),
           "T_settles_ms": round(t_settle, 3), "T_serial_ms": round(t_serial, 3),
           "S_ideal": round(s_ideal, 3)}
    best = None
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the settle kernel runs 3 CTAs per SM (80 registers x 256 threads), the
    # GEMM one: "k SMs" caps the pipe at 3k CTAs and the GEMM at SMs - k
    occ = 3
    for vname, pipe_cap, gemm_cap in (("all_sms", 0, 0), ("one_settle_cta_per_sm", sms, 0),
                                      ("pipe_38_sms", occ * 38, 0),
                                      ("partitioned_38_sms", occ * 38, sms - 38),
                                      ("partitioned_76_sms", occ * 76, sms - 76)):
        _, h = B.dp_settle_pipe_create(pipe_cap)
        B.dp_set_cta_limits(gemm_cap, 0)
        try:
            def push(g, l):
                t, cnt, gm = tables[g]
                B.dp_settle_pipe_push(h, t[l], cnt, K, gm, N, B.DP_BF16, accs[l], phase(g),
                                      o32, o16, 1.0 / K, sh)

            def per_group():
                for g in range(G):
                    for l in range(L):
                        gemm()
                    for l in range(L):
                        push(g, l)
                B.dp_settle_pipe_wait(h, sh)

            def per_layer():
                for g in range(G):
                    for l in range(L):
                        gemm()
                        push(g, l)
                B.dp_settle_pipe_wait(h, sh)

            for sname, fn in (("per_group", per_group), ("per_layer", per_layer)):
                tc = timed(fn)
                s_ = t_serial / tc
                r = {"T_ms": round(tc, 3), "S": round(s_, 3),
                     "pct_of_ideal": round(100 * (s_ - 1) / max(s_ideal - 1, 1e-9), 1)}
                out[f"{vname}_{sname}"] = r
                if best is None or s_ > best["S"]:
                    best = {"schedule": f"{vname}_{sname}", **r, "S_ideal": round(s_ideal, 3)}
        finally:
            B.dp_set_cta_limits(0, 0)
            B.dp_settle_pipe_destroy(h)
    out["best"] = best
    st = B.dp_get_device_error(sh)
    assert st == B.DP_OK, B.status_string(st)
    del accs, wl
    return out


def measure_ddp_overlap(dev, reps, cap_mb=25):
    """DDP's asynchronous bucket all-reduce beside the backward ("CMU 11-868
    L14-L15", "When to sync: gradient bucketing"): GPT-2-small fp32
    gradients on K=8 ranks in 25 MiB buckets; the backward of each bucket's
    layers is stood in for by one 4(b) GEMM (0.16 ms) before its parameters
    are marked ready in reverse order.  Serial: the Reducer launches every
    bucket on the caller's stream; overlap: on its own stream, joined before
    the optimizer step.  S and % of ideal as for the settle pipeline."""
    import torch

    from ring_allreduce_gradient_gb300 import binding as B
    from ring_allreduce_gradient_gb300.collectives import Reducer
    import workloads

    K = K_RANKS
    numels = workloads.gpt2_small_numels()
    grads = workloads.ddp_grads_device(numels, K, dev)
    red = Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=cap_mb * MiB, scale=1.0 / K)
    ptrs = [[grads[r][p].data_ptr() for r in range(K)] for p in range(len(numels))]
    P = len(numels)
    # the first parameter of each bucket in backward order (the highest index)
    opens = {max(p for p in range(P) if red.param_slot(p)[0] == b) for b in range(red.num_buckets)}
    wl = make_workload("agmm_b", dev, 0)
    x, ws_, y, wsp = wl["keep"]
    wsb = B.dp_allgather_matmul_workspace_size(8192, 4096, 8, 512)
    sa = torch.cuda.Stream(device=dev)
    sh = sa.cuda_stream

    def gemm():
        B.dp_allgather_matmul(x, 8192, 4096, ws_, 8, 512, y, B.DP_BF16, sh, workspace=wsp,
                              workspace_bytes=wsb)

    def iteration(with_gemm=True, with_ar=True):
        for p in reversed(range(P)):
            if with_gemm and p in opens:
                gemm()
            if with_ar:
                red.mark_ready(p, ptrs[p], sh)
        if with_ar:
            B.dp_reducer_wait(red.handle, sh)
            st, _ = red.finish()
            assert st == B.DP_OK

    def timed(fn):
        ts = []
        for i in range(reps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(sa)
            fn()
            b.record(sa)
            torch.cuda.synchronize()
            if i >= 2:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    t_gemm = timed(lambda: iteration(True, False))
    t_ar = timed(lambda: iteration(False, True))
    t_serial = timed(lambda: iteration(True, True))
    s_ideal = t_serial / max(t_gemm, t_ar)
    out = {"bucket_cap_mib": cap_mb, "buckets": red.num_buckets,
           "T_gemms_ms": round(t_gemm, 3), "T_allreduces_ms": round(t_ar, 3),
           "T_serial_ms": round(t_serial, 3), "S_ideal": round(s_ideal, 3),
           "note": "eager host-driven iteration (mark_ready per parameter); T_serial with "
                   "the default (bulk-copy) bucket kernel"}
    prev = B.dp_get_collective_variant()
    best = None
    for vname, variant in (("bulk_copy", 2), ("registers", 1)):
        B.dp_set_collective_variant(variant)
        red.set_overlap(True)
        try:
            t_over = timed(lambda: iteration(True, True))
        finally:
            red.set_overlap(False)
            B.dp_set_collective_variant(prev)
        s_ = t_serial / t_over
        r = {"T_overlap_ms": round(t_over, 3), "S": round(s_, 3),
             "pct_of_ideal": round(100 * (s_ - 1) / max(s_ideal - 1, 1e-9), 1)}
        out[f"overlap_{vname}"] = r
        if best is None or s_ > best["S"]:
            best = dict(r, kernel=vname)
    out.update({"T_serial_ms": round(t_serial, 3), "T_overlap_ms": best["T_overlap_ms"],
                "S": best["S"], "pct_of_ideal": best["pct_of_ideal"],
                "best_kernel": best["kernel"]})
    st = B.dp_get_device_error(sh)
    assert st == B.DP_OK, B.status_string(st)
    del grads, red, wl
    return out


# ----------------------------------------------------------------------------
# collective || GEMM on two streams (NEXT rows: settle overlap, copy engines)
# ----------------------------------------------------------------------------

def measure_c3(dev, reps=20):
    """Speedup of running a collective concurrently with the tensor-core GEMM.

    "Optimizing ML Concurrent Computation and Communication with GPU DMA
    Engines", Problem Formulation: S = T_serial / T_concurrent with
    T_serial = T_GEMM + T_comm and S_ideal = T_serial / max(T_GEMM, T_comm);
    "% of ideal" = (S - 1) / (S_ideal - 1).  GEMM: x[8192,4096] . w^T with the
    weight gathered from 8 shards.  Collectives: the FSDP parameter all-gather
    (8 shards x 16 MiB fp32 -> 8 x 128 MiB) on the SMs or on the copy engines,
    and the gradient settle (the headline reduce-scatter).  Variants: base
    (GEMM launched first), priority (collective first, on a high-priority
    stream), partitioned (GEMM limited to SMs-k CTAs, the collective to k CTAs:
    every kernel here runs one CTA per SM, so the two share the SMs exactly).
    """
    import torch

    from ring_allreduce_gradient_gb300 import binding as B
    import workloads

    K = K_RANKS
    sa = torch.cuda.Stream(device=dev)
    sb_lo = torch.cuda.Stream(device=dev)
    sb_hi = torch.cuda.Stream(device=dev, priority=-1)
    g = torch.Generator(device=dev)
    g.manual_seed(40)
    M, D, Fs = 8192, 4096, 512
    x = (torch.randn(M, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    ws_ = [(torch.randn(Fs, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
           for _ in range(K)]
    y = torch.empty(M, K * Fs, dtype=torch.bfloat16, device=dev)
    C = 16 * MiB // 4
    shards = [torch.randn(C, device=dev) for _ in range(K)]
    outs = [torch.empty(K * C, device=dev) for _ in range(K)]
    N = N_ELEMS
    grads = workloads.fsdp_grads_device(K, N, dev)
    o32 = [torch.empty(N // K, device=dev) for _ in range(K)]
    o16 = [torch.empty(N // K, dtype=torch.bfloat16, device=dev) for _ in range(K)]

    def gemm(s):
        B.dp_allgather_matmul(x, M, D, ws_, K, Fs, y, B.DP_BF16, s.cuda_stream)

    comms = {
        "allgather_sm": lambda s: B.dp_all_gather(shards, K, C, B.DP_FP32, outs, s.cuda_stream),
        "allgather_copy_engine": lambda s: B.dp_all_gather_copy_engine(shards, K, C, B.DP_FP32,
                                                                       outs, s.cuda_stream),
        "settle_reduce_scatter": lambda s: B.dp_reduce_scatter_dual(
            grads, K, N, B.DP_BF16, o32, o16, 1.0 / K, s.cuda_stream),
    }

    def alone(fn, s):
        for _ in range(3):
            fn(s)
        torch.cuda.synchronize()
        return statistics.median(time_events(lambda: fn(s), reps, s))

    def together(comm, first_comm, sb):
        ts = []
        for i in range(reps + 3):
            e0, ea, eb = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(sa)
            sb.wait_event(e0)
            if first_comm:
                comm(sb)
                gemm(sa)
            else:
                gemm(sa)
                comm(sb)
            eb.record(sb)
            sa.wait_event(eb)
            ea.record(sa)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(ea))
        return statistics.median(ts)

    res = {}
    try:
        for cname, comm in comms.items():
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            variants = [("base", False, sb_lo, (0, 0)), ("priority", True, sb_hi, (0, 0))]
            variants += [(f"partitioned_k{k}", True, sb_hi, (sms - k, k)) for k in (16, 38, 76)]
            if cname == "allgather_copy_engine":
                variants = variants[:2]
            out = {}
            for vname, first, sb, lim in variants:
                B.dp_set_cta_limits(*lim)
                tg = alone(gemm, sa)
                tc = alone(comm, sb)
                tcc = together(comm, first, sb)
                ser = tg + tc
                s_ = ser / tcc
                s_ideal = ser / max(tg, tc)
                out[vname] = {"T_gemm_ms": round(tg, 4), "T_comm_ms": round(tc, 4),
                              "T_concurrent_ms": round(tcc, 4), "S": round(s_, 3),
                              "S_ideal": round(s_ideal, 3),
                              "pct_of_ideal": round(100 * (s_ - 1) / max(s_ideal - 1, 1e-9), 1)}
            res[cname] = out
    finally:
        B.dp_set_cta_limits(0, 0)
    st = B.dp_get_device_error(sa.cuda_stream)
    assert st == B.DP_OK, B.status_string(st)
    return res


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
    ap.add_argument("--workload", choices=["rs", "ar", "ag", "agmm_b", "agmm_a", "odc", "tp_ar",
                                           "tp_rs", "tp_rs_xw", "tp_fixture", "wgrad", "ddp1",
                                           "ddp25", "ddp100"],
                    default="rs", help="rs (the headline) or one other row on its own")
    ap.add_argument("--no-rows", action="store_true", help="skip the other rows' measurements")
    ap.add_argument("--c3-only", action="store_true",
                    help="print only the collective || GEMM concurrency measurements")
    ap.add_argument("--pipeline-only", action="store_true",
                    help="print only the settle pipeline measurements (variable-length workload)")
    ap.add_argument("--ddp-overlap-only", action="store_true",
                    help="print only the DDP overlap measurement")
    ap.add_argument("--sweep-only", action="store_true",
                    help="print only the all-reduce bandwidth sweep")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--row-reps", type=int, default=20)
    ap.add_argument("--odc-layers", type=int, default=32)
    ap.add_argument("--ar-mib", type=int, default=1024, help="all-reduce workload: MiB per rank")
    ap.add_argument("--variant", type=int, default=0, choices=[0, 1, 2],
                    help="all-reduce/all-gather implementation: 0 auto, 1 registers, 2 bulk copies")
    ap.add_argument("--cpu-sample-mib", type=int, default=64,
                    help="per-rank elements (Mi) of the oracle's timed sample")
    ap.add_argument("--ref-sample-mib", type=int, default=4)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, _, _ = dist_env()
    if ws != args.gpus and not (ws == 1 and args.gpus == 1):
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={ws}", file=sys.stderr)
    if args.sweep_only:
        import torch
        torch.cuda.set_device(0)
        from ring_allreduce_gradient_gb300 import binding as B
        from ring_allreduce_gradient_gb300 import build as cuda_build
        cuda_build.build()
        B.load()
        print(json.dumps({"allreduce_sweep": measure_sweep(torch.device("cuda", 0),
                                                           peaks()[0])}), flush=True)
    elif args.pipeline_only:
        import torch
        torch.cuda.set_device(0)
        from ring_allreduce_gradient_gb300 import binding as B
        from ring_allreduce_gradient_gb300 import build as cuda_build
        cuda_build.build()
        B.load()
        dev = torch.device("cuda", 0)
        wl = make_workload("odc", dev, 0, args.odc_layers)
        grads = wl["keep"][0]
        m = wl["cfg"]["microbatches"]
        print(json.dumps({"settle_pipeline": measure_settle_pipeline(
            dev, grads, m, args.odc_layers, 16 * MiB, max(3, args.row_reps // 4))}), flush=True)
    elif args.ddp_overlap_only:
        import torch
        torch.cuda.set_device(0)
        from ring_allreduce_gradient_gb300 import binding as B
        from ring_allreduce_gradient_gb300 import build as cuda_build
        cuda_build.build()
        B.load()
        print(json.dumps({"ddp_overlap": measure_ddp_overlap(torch.device("cuda", 0),
                                                             max(3, args.row_reps // 4))}),
              flush=True)
    elif args.c3_only:
        import torch
        torch.cuda.set_device(0)
        from ring_allreduce_gradient_gb300 import binding as B
        from ring_allreduce_gradient_gb300 import build as cuda_build
        cuda_build.build()
        B.load()
        print(json.dumps({"c3": measure_c3(torch.device("cuda", 0))}), flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
