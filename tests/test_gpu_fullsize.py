"""GPU parity at the benchmark's full sizes, in its launch configuration, for
the rows whose other tests run smaller: the all-gather (8 shards of 32 MiB),
the tensor-parallel GEMM all-reduce (8 x (8192x512 . 512x4096)), and the DDP
bucketed all-reduce of GPT-2-small-shaped gradients (124M parameters in 148
tensors, 25 MiB buckets).

Where the oracle cannot run the whole problem in seconds, outputs are checked
through properties that hold at any size (the all-gather is a copy; every
all-reduce copy is the same; the reduce-scatter is the all-reduce's rows) or
sampled elements are computed by the oracle one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
MiB = 1024 * 1024


def test_all_gather_bench_config_is_the_concatenation():
    # "CMU 11-868 L14-L15", section "Ring AllReduce: ReduceScatter, then
    # AllGather": after the all-gather every rank holds every finished chunk
    K, C = 8, 32 * MiB // 4
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    shards = [torch.randn(C, generator=g, device=DEV) for _ in range(K)]
    outs = col.all_gather(shards)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    want = torch.cat(shards).view(torch.int32)
    for r in range(K):
        assert torch.equal(outs[r].view(torch.int32), want)


def test_tp_allreduce_bench_config_copies_and_rows():
    # every rank's copy is bitwise the same, and row shard c of the fused
    # reduce-scatter (checked against the fp64 oracle elsewhere) is bitwise
    # rows [c M/K, (c+1) M/K) of it
    K, M, Ds, F = 8, 8192, 512, 4096
    g = torch.Generator(device=DEV)
    g.manual_seed(60)
    xs = [(torch.randn(M, Ds, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
          for _ in range(K)]
    ws = [(torch.randn(F, Ds, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
          for _ in range(K)]
    ys = col.matmul_allreduce(xs, ws, 1.0, torch.bfloat16)
    shards = col.matmul_reduce_scatter(xs, ws, 1.0, torch.bfloat16)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    y0 = ys[0].view(torch.int16)
    for r in range(1, K):
        assert torch.equal(ys[r].view(torch.int16), y0)
    rows = M // K
    for c in range(K):
        assert torch.equal(shards[c].view(torch.int16), y0[c * rows:(c + 1) * rows])
    assert float(ys[0].float().abs().mean()) > 0


def _bucket_samples(C, n, rng, count=160):
    """Offsets inside a bucket of n elements with chunk length C: the chunk
    edges on both sides, the ends, and random ones."""
    edges = [0, n - 1]
    for c in range(1, (n + C - 1) // C):
        edges += [c * C - 1, c * C, min(c * C + 1, n - 1)]
    pts = np.unique(np.concatenate([np.array(edges, np.int64), rng.integers(0, n, count)]))
    return pts[(pts >= 0) & (pts < n)]


@pytest.mark.parametrize("overlap", [False, True])
def test_ddp_bench_config_sampled(overlap):
    # one Reducer iteration over GPT-2-small-shaped fp32 gradients on 8 ranks
    # (25 MiB buckets, parameters ready in backward order), as the benchmark
    # runs it -- with the buckets on the caller's stream, or on the Reducer's
    # own stream (overlap mode) joined before the check; sampled elements of
    # every bucket against the oracle's ring fold of that bucket, bit for
    # bit, on every rank
    K = 8
    numels = workloads.gpt2_small_numels()
    grads = workloads.ddp_grads_device(numels, K, DEV)
    red = col.Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=25 * MiB, scale=1.0 / K)
    if overlap:
        red.set_overlap(True)
    rng = np.random.default_rng(17)

    # bucket b: its parameters and their offsets, then the sampled positions
    slots = [red.param_slot(p) for p in range(len(numels))]
    plan = []
    for b in range(red.num_buckets):
        _, n = red.bucket_info(b)
        members = sorted((off, p) for p, (bb, off) in enumerate(slots) if bb == b)
        C = (n + K - 1) // K
        pts = _bucket_samples(C, n, rng)
        starts = np.array([off for off, _ in members], np.int64)
        which = np.searchsorted(starts, pts, side="right") - 1
        loc = [(members[w][1], int(q - members[w][0])) for w, q in zip(which, pts)]
        plan.append((n, C, pts, loc))

    def gather(plan_entry):
        _, _, _, loc = plan_entry
        out = np.empty((K, len(loc)), np.float32)
        by_param = {}
        for i, (p, j) in enumerate(loc):
            by_param.setdefault(p, []).append((i, j))
        for p, lst in by_param.items():
            idx = torch.tensor([j for _, j in lst], device=DEV)
            pos = [i for i, _ in lst]
            for r in range(K):
                out[r, pos] = grads[r][p][idx].cpu().numpy()
        return out

    inputs = [gather(e) for e in plan]

    ptrs = [[grads[r][p].data_ptr() for r in range(K)] for p in range(len(numels))]
    for p in reversed(range(len(numels))):
        red.mark_ready(p, ptrs[p])
    if overlap:
        red.wait()
    st, first_pending = red.finish()
    assert st == B.DP_OK and first_pending == -1
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK

    for (n, C, pts, loc), vals in zip(plan, inputs):
        S = len(pts)
        # sample s goes to offset s of its own chunk c_s in K buffers of K*S
        # elements, so the oracle folds it in chunk c_s's ring order
        chunks = pts // C
        bufs = [np.zeros(K * S, np.float32) for _ in range(K)]
        for r in range(K):
            bufs[r][chunks * S + np.arange(S)] = vals[r]
        s32, _ = oracle.reduce_scatter(bufs, 1.0 / K)
        want = np.array([s32[c][s] for s, c in enumerate(chunks)], np.float32)
        got = gather((n, C, pts, loc))
        for r in range(K):
            assert np.array_equal(got[r].view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------
# element counts past 2^31: 64-bit offsets in every streaming kernel
# ---------------------------------------------------------------------------

BIG = (1 << 31) + 64  # elements per rank


def _sample(N, C, rng):
    edges = [0, C - 1, C, N - 1, (1 << 31) - 1, 1 << 31, (1 << 31) + 1]
    return np.unique(np.concatenate([rng.integers(0, N, 1024), np.array(edges, np.int64)]))


@pytest.mark.parametrize("variant", [1, 2])
def test_all_reduce_past_2_31_elements_sampled(variant):
    """K=2 x (2^31 + 64) fp32 per rank, in place (16 GiB), both kernels:
    sampled elements around the 2^31 boundary and the chunk boundary against
    the oracle's ring fold of the same elements."""
    K, N = 2, BIG
    C = N // K
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    bufs = [torch.rand(N, generator=g, device=DEV) * 2 - 1 for _ in range(K)]
    idx = _sample(N, C, np.random.default_rng(3))
    it = torch.from_numpy(idx).to(DEV)
    vals = torch.stack([b[it] for b in bufs]).cpu().numpy()
    B.dp_set_collective_variant(variant)
    try:
        col.all_reduce_(bufs, 0.5)
        torch.cuda.synchronize()
    finally:
        B.dp_set_collective_variant(0)
    assert B.dp_get_device_error() == B.DP_OK
    S = idx.size
    small = [np.zeros(K * S, np.float32) for _ in range(K)]
    for r in range(K):
        small[r][(idx // C) * S + np.arange(S)] = vals[r]
    r32, _ = oracle.reduce_scatter(small, 0.5, ("f32",))
    want = np.array([r32[int(e) // C][s] for s, e in enumerate(idx)], np.float32)
    for r in range(K):
        assert np.array_equal(bufs[r][it].cpu().numpy().view(np.uint32), want.view(np.uint32))
    del bufs
    torch.cuda.empty_cache()


def test_reduce_scatter_past_2_31_elements_sampled():
    """K=2 x (2^31 + 64) bf16 per rank -> fp32 + bf16 shards of 2^30 + 32."""
    K, N = 2, BIG
    C = N // K
    g = torch.Generator(device=DEV)
    g.manual_seed(12)
    bufs = [(torch.randn(N, generator=g, device=DEV) * 1e-3).to(torch.bfloat16) for _ in range(K)]
    idx = _sample(N, C, np.random.default_rng(4))
    it = torch.from_numpy(idx).to(DEV)
    vals = [workloads.torch_bf16_to_bits(b[it]) for b in bufs]
    o32, o16 = col.reduce_scatter(bufs, 1.0 / K)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    S = idx.size
    small = [np.zeros(K * S, np.uint16) for _ in range(K)]
    for r in range(K):
        small[r][(idx // C) * S + np.arange(S)] = vals[r]
    r32, r16 = oracle.reduce_scatter(small, 1.0 / K)
    for s, e in enumerate(idx):
        c, o = int(e) // C, int(e) % C
        assert o32[c][o].view(torch.int32).item() == int(r32[c][s].view(np.int32)), e
        assert int(workloads.torch_bf16_to_bits(o16[c][o:o + 1])[0]) == int(r16[c][s]), e
    del bufs, o32, o16
    torch.cuda.empty_cache()


def test_all_gather_past_2_31_elements_is_the_concatenation():
    """K=2 shards of 2^30 + 32 fp32 -> 2 x (2^31 + 64): both schedules of the
    bulk-copy kernel (the whole GPU, and under a CTA cap)."""
    K, C = 2, BIG // 2
    g = torch.Generator(device=DEV)
    g.manual_seed(13)
    shards = [torch.randn(C, generator=g, device=DEV) for _ in range(K)]
    saved = B.dp_get_cta_limits()
    try:
        for cap in (0, 40):
            B.dp_set_cta_limits(saved[0], cap)
            outs = col.all_gather(shards)
            torch.cuda.synchronize()
            assert B.dp_get_device_error() == B.DP_OK
            for r in range(K):
                for c in range(K):
                    assert torch.equal(outs[r][c * C:(c + 1) * C].view(torch.int32),
                                       shards[c].view(torch.int32)), (cap, r, c)
            del outs
    finally:
        B.dp_set_cta_limits(*saved)
    del shards
    torch.cuda.empty_cache()
