"""GPU parity of the cross-iteration settle pipeline ("Using ODC to Accelerate
AMD SFT Training", section "Discussion: Settle Does Not Yet Overlap with
Backward"): group settles (dp_odc_settle_group) and the pipe that runs them
on its own stream beside the caller's compute (dp_settle_pipe_*), bit for
bit against the oracle's pipelined settle; the GEMMs that produce the
gradients against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def f32bits(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def host_grads(K, N, m, seed, dt="bf16"):
    rng = np.random.default_rng(seed)
    out = []
    for r in range(K):
        row = []
        for j in range(m[r]):
            g = rng.standard_normal(N).astype(np.float32) * np.float32(1e-3 * (1 + j))
            row.append(workloads.to_bf16_bits(g) if dt == "bf16" else g)
        out.append(row)
    return out


def to_dev(a):
    if a.dtype == np.uint16:
        return workloads.bits_to_torch_bf16(a).to(DEV)
    return torch.from_numpy(a).to(DEV)


def group_slices(rows, bounds):
    """rows[r] is rank r's microbatch list; group g is j in [bounds[g], bounds[g+1])."""
    return [[row[lo:hi] for row in rows] for lo, hi in zip(bounds[:-1], bounds[1:])]


def phase_of(g, G):
    return (B.DP_SETTLE_FIRST if g == 0 else 0) | (B.DP_SETTLE_LAST if g == G - 1 else 0)


def check_against_oracle(o32, o16, hg, m, bounds, scale, N, dt):
    e32, e16 = oracle.odc_pipelined(hg, m, bounds, scale, N,
                                    grad_dtype=oracle.BF16 if dt == "bf16" else oracle.F32)
    K = len(hg)
    for c in range(K):
        assert np.array_equal(f32bits(o32[c]), e32[c].view(np.uint32)), c
        assert np.array_equal(workloads.torch_bf16_to_bits(o16[c]), e16[c]), c


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("N", [8 * 8 * 700, 8 * 1001])
@pytest.mark.parametrize("bounds", [[0, 2, 5, 8], [0, 8], [0, 1, 2, 3, 4, 5, 6, 7, 8],
                                    [0, 3, 3, 8]])
def test_group_settles_match_the_oracle(dt, N, bounds):
    """Group after group on one stream (vector path for N = 8*8*700, scalar
    path for chunks of 1001 elements), an empty group included."""
    K = 8
    m, _ = workloads.odc_schedule(K)
    m = [int(v) for v in m]
    hg = host_grads(K, N, m, 41, dt)
    dg = [[to_dev(g) for g in row] for row in hg]
    gdt = torch.bfloat16 if dt == "bf16" else torch.float32
    C = N // K
    acc = [torch.full((C,), 777.0, device=DEV) for _ in range(K)]
    o32 = [torch.full((C,), float("nan"), device=DEV) for _ in range(K)]
    o16 = [torch.full((C,), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    groups = group_slices(dg, bounds)
    for g, grp in enumerate(groups):
        col.odc_settle_group(grp, N, acc, phase_of(g, len(groups)), 1.0 / K, out=(o32, o16),
                             grad_dtype=gdt)
    torch.cuda.synchronize()
    check_against_oracle(o32, o16, hg, m, bounds, 1.0 / K, N, dt)
    if len(groups) == 1:  # one group is the one-settle call, bit for bit
        a32, a16 = col.odc_reduce_scatter(dg, m, N, 1.0 / K, gdt)
        for c in range(K):
            assert torch.equal(a32[c].view(torch.int32), o32[c].view(torch.int32))
            assert torch.equal(a16[c].view(torch.int16), o16[c].view(torch.int16))
    assert B.dp_get_device_error() == B.DP_OK


def test_group_settle_by_hand():
    """The hand-worked binary32 values of the pipeline pin, on the GPU, at the
    pin's size (scalar path) and with every chunk repeated 1024 times."""
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "odc_pipeline_k2.txt")
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    K, N0 = map(int, rows[0].split())
    per_rank = [[float(v) for v in rows[1 + r].split()] for r in range(K)]
    for rep in (1, 1024):
        N = N0 * rep
        dg = [[torch.full((N,), v, dtype=torch.bfloat16, device=DEV) for v in vals]
              for vals in per_rank]
        for line in rows[1 + K:-1]:
            bnd, exp = line.split(";")
            bounds = [int(v) for v in bnd.split()]
            exp = [float(v) for v in exp.split()]
            acc = [torch.empty(N // K, device=DEV) for _ in range(K)]
            o32 = [torch.empty(N // K, device=DEV) for _ in range(K)]
            o16 = [torch.empty(N // K, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
            groups = group_slices(dg, bounds)
            for g, grp in enumerate(groups):
                col.odc_settle_group(grp, N, acc, phase_of(g, len(groups)), 1.0,
                                     out=(o32, o16))
            for c in range(K):
                want = torch.full((N // K,), exp[c])
                assert torch.equal(o32[c].cpu(), want), (bounds, c)
                assert torch.equal(o16[c].float().cpu(), want), (bounds, c)


def _gemm_grads(K, m, M, D, Fs, seed):
    """Per (rank, microbatch) GEMM operands: x_{r,j}[M, D] and one set of 8
    weight shards w_k[Fs, D]; the product y = x . w^T ([M, 8*Fs] bf16) is that
    microbatch's gradient (N = M * 8 * Fs elements)."""
    xs = [[workloads.to_bf16_bits(np.random.default_rng(seed + 100 * r + j)
                                  .standard_normal((M, D), dtype=np.float32) * np.float32(0.02))
           for j in range(m[r])] for r in range(K)]
    _, ws = workloads.gemm_operands(16, D, 8, Fs)
    return xs, ws


@pytest.mark.parametrize("cta_limit", [0, 16])
def test_pipe_settles_beside_the_gemms_that_produce_the_gradients(cta_limit):
    """The schedule of the page: group g's backward (here the GEMMs that
    write group g's microbatch gradients) on the caller's stream, group g's
    settle pushed to the pipe, group g+1's GEMMs enqueued right behind it,
    one join at the end.  The settle reads what the GEMMs wrote: its result
    is bit-exact against the oracle's pipelined settle of the GEMM outputs
    (copied back after the join), and the GEMMs are within the fp64
    tolerance of the oracle."""
    K = 8
    m = [2, 3, 1, 3, 2, 1, 3, 2]
    bounds = [0, 1, 2, 3]
    M, D, Fs = 512, 512, 64
    N = M * 8 * Fs
    xs_h, ws_h = _gemm_grads(K, m, M, D, Fs, 50)
    xs = [[workloads.bits_to_torch_bf16(x).to(DEV) for x in row] for row in xs_h]
    ws = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws_h]
    ys = [[torch.full((M, 8 * Fs), float("nan"), dtype=torch.bfloat16, device=DEV)
           for _ in range(m[r])] for r in range(K)]
    pipe = col.SettlePipe(K, N, DEV, cta_limit=cta_limit)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    G = len(bounds) - 1
    with torch.cuda.stream(s):
        for g in range(G):
            lo, hi = bounds[g], bounds[g + 1]
            for r in range(K):
                for j in range(lo, min(hi, m[r])):
                    B.dp_allgather_matmul(xs[r][j], M, D, ws, 8, Fs, ys[r][j], B.DP_BF16, s)
            grp = [[ys[r][j] for j in range(lo, min(hi, m[r]))] for r in range(K)]
            pipe.push(grp, first=(g == 0), last=(g == G - 1), scale=1.0 / K, stream=s)
        pipe.wait(stream=s)
    s.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    hy = [[workloads.torch_bf16_to_bits(y.reshape(-1)) for y in row] for row in ys]
    check_against_oracle(pipe.out32, pipe.out16, hy, m, bounds, 1.0 / K, N, "bf16")
    for r, j in ((0, 0), (1, 2), (7, 1)):
        ref = oracle.allgather_matmul_f64(xs_h[r][j], ws_h)
        got = ys[r][j].double().cpu().numpy()
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2
    pipe.close()


def test_pipe_in_a_cuda_graph_replays_to_the_same_bits():
    """Pushes and the join captured in a CUDA graph (the pipe's stream forks
    from and joins the capturing stream); two replays give the eager bits."""
    K, N = 8, 8 * 8 * 512
    m = [3, 1, 2, 4, 2, 1, 3, 2]
    bounds = [0, 2, 4]
    hg = host_grads(K, N, m, 43)
    dg = [[to_dev(g) for g in row] for row in hg]
    groups = group_slices(dg, bounds)
    pipe = col.SettlePipe(K, N, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # eager once (also sets the kernels' attributes up)
        for g, grp in enumerate(groups):
            pipe.push(grp, first=(g == 0), last=(g == len(groups) - 1), scale=1.0 / K, stream=s)
        pipe.wait(stream=s)
    s.synchronize()
    e32 = [t.clone() for t in pipe.out32]
    check_against_oracle(pipe.out32, pipe.out16, hg, m, bounds, 1.0 / K, N, "bf16")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for g, grp in enumerate(groups):
            pipe.push(grp, first=(g == 0), last=(g == len(groups) - 1), scale=1.0 / K, stream=s)
        pipe.wait(stream=s)
    for _ in range(2):
        for t in pipe.out32:
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for c in range(K):
            assert torch.equal(pipe.out32[c].view(torch.int32), e32[c].view(torch.int32))
    assert B.dp_get_device_error() == B.DP_OK
    pipe.close()


def test_pipe_pushes_from_two_threads_keep_each_pipe_consistent():
    """Two pipes driven from two host threads at once, each on its own
    stream: both results bit-exact against the oracle."""
    import threading
    K, N = 8, 8 * 8 * 256
    cases = []
    for seed, m, bounds in ((44, [2, 2, 1, 3, 1, 2, 2, 1], [0, 1, 3]),
                            (45, [1, 3, 2, 2, 3, 1, 1, 2], [0, 2, 3])):
        hg = host_grads(K, N, m, seed)
        dg = [[to_dev(g) for g in row] for row in hg]
        cases.append((hg, dg, m, bounds, col.SettlePipe(K, N, DEV), torch.cuda.Stream()))
    torch.cuda.synchronize()
    errs = []

    def run(case):
        try:
            torch.cuda.set_device(0)
            hg, dg, m, bounds, pipe, s = case
            groups = group_slices(dg, bounds)
            for _ in range(3):
                for g, grp in enumerate(groups):
                    pipe.push(grp, first=(g == 0), last=(g == len(groups) - 1),
                              scale=1.0 / K, stream=s)
                pipe.wait(stream=s)
            s.synchronize()
        except Exception as e:  # reported below
            errs.append(e)

    th = [threading.Thread(target=run, args=(c,)) for c in cases]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errs, errs
    for hg, dg, m, bounds, pipe, s in cases:
        check_against_oracle(pipe.out32, pipe.out16, hg, m, bounds, 1.0 / K, N, "bf16")
        pipe.close()
    assert B.dp_get_device_error() == B.DP_OK


def test_pipe_full_layer_sampled():
    """One layer of the variable-length workload at full size (K=8, 16 Mi
    elements, the microbatch schedule and token scales of the benchmark,
    gradients drawn on the device) through the pipe with the benchmark's two
    groups (j < 4, j >= 4): sampled elements bit-exact against the oracle's
    pipelined settle of the same elements (each sample placed in its chunk
    of a small problem, so its ring order is the same)."""
    K, N = 8, 16 * workloads.MiB
    C = N // K
    m, toks = workloads.odc_schedule(K)
    m = [int(v) for v in m]
    bounds = [0, 4, max(max(m), 4)]
    layer = 5
    dg = [[workloads.odc_grad(layer, r, j, N, int(toks[r, j]), DEV) for j in range(m[r])]
          for r in range(K)]
    pipe = col.SettlePipe(K, N, DEV)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    groups = group_slices(dg, bounds)
    with torch.cuda.stream(s):
        for g, grp in enumerate(groups):
            pipe.push(grp, first=(g == 0), last=(g == len(groups) - 1), scale=1.0 / K, stream=s)
        pipe.wait(stream=s)
    s.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    rng = np.random.default_rng(7)
    idx = np.unique(np.concatenate([rng.integers(0, N, 1024), [0, C - 1, C, N - 1]]))
    it = torch.from_numpy(idx).to(DEV)
    S = idx.size
    small = []
    for r in range(K):
        row = []
        for j in range(m[r]):
            buf = np.zeros(K * S, np.uint16)
            buf[(idx // C) * S + np.arange(S)] = workloads.torch_bf16_to_bits(dg[r][j][it])
            row.append(buf)
        small.append(row)
    e32, e16 = oracle.odc_pipelined(small, m, bounds, 1.0 / K, K * S)
    got32 = np.stack([f32bits(pipe.out32[c]) for c in range(K)])
    got16 = np.stack([workloads.torch_bf16_to_bits(pipe.out16[c]) for c in range(K)])
    for q, e in enumerate(idx):
        c, i = divmod(int(e), C)
        assert got32[c, i] == e32[c][q].view(np.uint32), e
        assert got16[c, i] == e16[c][q], e
    pipe.close()


@pytest.mark.parametrize("K,m,bounds,N", [
    (1, [5], [0, 2, 5], 8 * 512),            # one rank: the owner adds its own group sums
    (16, [1 + (r * 7) % 16 for r in range(16)], [0, 5, 10, 16], 16 * 8 * 64),
    (3, [2, 4, 1], [0, 1, 4], 3 * 1001),     # an odd rank count, ragged chunks
])
def test_group_settles_edge_ranks(K, m, bounds, N):
    hg = host_grads(K, N, m, 47)
    dg = [[to_dev(g) for g in row] for row in hg]
    C = N // K
    acc = [torch.empty(C, device=DEV) for _ in range(K)]
    o32 = [torch.empty(C, device=DEV) for _ in range(K)]
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    groups = group_slices(dg, bounds)
    for g, grp in enumerate(groups):
        col.odc_settle_group(grp, N, acc, phase_of(g, len(groups)), 1.0 / K, out=(o32, o16))
    torch.cuda.synchronize()
    check_against_oracle(o32, o16, hg, m, bounds, 1.0 / K, N, "bf16")


def test_group_settle_unaligned_accumulator_and_noops():
    """An owner accumulator 4 bytes off a 16-byte boundary takes the scalar
    path with the same bits; N == 0 launches nothing; the whole-minibatch
    phase needs no accumulator."""
    K, N = 4, 4 * 8 * 96
    m = [2, 3, 1, 2]
    bounds = [0, 1, 3]
    hg = host_grads(K, N, m, 48)
    dg = [[to_dev(g) for g in row] for row in hg]
    C = N // K
    raw = [torch.empty(C + 1, device=DEV) for _ in range(K)]
    acc = [t[1:] for t in raw]
    o32 = [torch.empty(C, device=DEV) for _ in range(K)]
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    groups = group_slices(dg, bounds)
    for g, grp in enumerate(groups):
        col.odc_settle_group(grp, N, acc, phase_of(g, len(groups)), 0.25, out=(o32, o16))
    torch.cuda.synchronize()
    check_against_oracle(o32, o16, hg, m, bounds, 0.25, N, "bf16")
    table = [g for row in dg for g in row[:1]]
    assert B.dp_odc_settle_group(table, [1] * K, K, 1, 0, B.DP_BF16, acc, 0, None, None, 1.0,
                                 check=False) == B.DP_OK
    w32, w16 = col.odc_reduce_scatter([row[:1] for row in dg], [1] * K, N, 0.25)
    assert B.dp_odc_settle_group(table, [1] * K, K, 1, N, B.DP_BF16, None,
                                 B.DP_SETTLE_FIRST | B.DP_SETTLE_LAST, o32, o16, 0.25) == B.DP_OK
    torch.cuda.synchronize()
    for c in range(K):
        assert torch.equal(o32[c].view(torch.int32), w32[c].view(torch.int32))


@pytest.mark.parametrize("K,dt", [(16, "f32"), (5, "bf16")])
def test_pipe_fp32_gradients_and_other_rank_counts(K, dt):
    """Through the pipe with fp32 gradients and sixteen ranks, and with an
    odd rank count and a ragged chunk length (scalar path)."""
    N = K * 8 * 96 if dt == "f32" else K * 1003
    m = [1 + (3 * r) % 5 for r in range(K)]
    bounds = [0, 2, 5]
    hg = host_grads(K, N, m, 49, dt)
    dg = [[to_dev(g) for g in row] for row in hg]
    gdt = torch.float32 if dt == "f32" else torch.bfloat16
    pipe = col.SettlePipe(K, N, DEV)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    groups = group_slices(dg, bounds)
    with torch.cuda.stream(s):
        for g, grp in enumerate(groups):
            pipe.push(grp, first=(g == 0), last=(g == len(groups) - 1), scale=1.0 / K,
                      grad_dtype=gdt, stream=s)
        pipe.wait(stream=s)
    s.synchronize()
    check_against_oracle(pipe.out32, pipe.out16, hg, m, bounds, 1.0 / K, N, dt)
    pipe.close()
