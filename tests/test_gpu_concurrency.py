"""Copy-engine all-gather, CTA limits and concurrent streams: results must be
bit-identical to the plain single-stream runs (and to the oracle)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def ibits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("K,C,dt,off", [(8, 4 * 4096, "f32", 0), (2, 1001, "bf16", 0),
                                        (8, 333, "f32", 1), (16, 8 * 77, "bf16", 0),
                                        (1, 5, "f32", 0), (3, 1, "bf16", 1)])
def test_copy_engine_all_gather_matches_oracle(K, C, dt, off):
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    rng = np.random.default_rng(K + C)
    host = [rng.uniform(-1, 1, C).astype(np.float32) for _ in range(K)]
    if dt == "bf16":
        host = [workloads.to_bf16_bits(h) for h in host]
    shards = []
    for h in host:
        t = workloads.bits_to_torch_bf16(h) if dt == "bf16" else torch.from_numpy(h)
        raw = torch.empty(C + off, dtype=tdt, device=DEV)
        raw[off:].copy_(t)
        shards.append(raw[off:])
    outs = [torch.empty(K * C + off, dtype=tdt, device=DEV)[off:] for _ in range(K)]
    B.dp_all_gather_copy_engine(shards, K, C, tdt, outs)
    ref = oracle.all_gather(host)
    kern = col.all_gather(shards)
    helper = col.all_gather(shards, copy_engines=True)
    for r in range(K):
        got = ibits(outs[r].cpu()).numpy()
        want = ref[r].view(np.int16) if dt == "bf16" else ref[r].view(np.int32)
        assert np.array_equal(got, want)
        assert torch.equal(ibits(outs[r]), ibits(kern[r]))
        assert torch.equal(ibits(outs[r]), ibits(helper[r]))


def test_cta_limits_leave_results_unchanged():
    K, N = 8, 8 * 8 * 3001
    bufs = workloads.fsdp_grads_device(K, N, DEV)
    x, ws = workloads.gemm_operands(512, 512, 8, 64)
    xd = workloads.bits_to_torch_bf16(x).to(DEV)
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    ar_in = [b.float() for b in bufs]

    def run():
        o32, o16 = col.reduce_scatter(bufs, 1.0 / K)
        y = col.allgather_matmul(xd, wd, torch.float32)
        ag = col.all_gather(o32)
        ar = [t.clone() for t in ar_in]
        col.all_reduce_(ar, 1.0 / K)
        torch.cuda.synchronize()
        return o32 + o16 + [y] + ag + ar

    ref = run()
    try:
        for g, s in [(1, 1), (40, 16), (150, 3)]:
            B.dp_set_cta_limits(g, s)
            assert B.dp_get_cta_limits() == (g, s)
            got = run()
            for a, b in zip(ref, got):
                assert torch.equal(ibits(a), ibits(b))
    finally:
        B.dp_set_cta_limits(0, 0)
    assert B.dp_get_device_error() == B.DP_OK


def test_gemm_and_settle_on_two_streams_concurrently():
    """The settle (reduce-scatter) on one stream while the GEMM runs on
    another: the settle's shards are bit-exact against the oracle's ring
    reduce-scatter on sampled elements (and equal to the serial run), the
    GEMM is within the fp64 tolerance of the oracle's product on sampled
    entries (and equal to the serial run bit for bit)."""
    K, N = 8, 8 * 1024 * 1024
    C = N // K
    bufs = workloads.fsdp_grads_device(K, N, DEV)
    M, D, Fs = 2048, 2048, 256
    x, ws = workloads.gemm_operands(M, D, 8, Fs)
    xd = workloads.bits_to_torch_bf16(x).to(DEV)
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    s32, s16 = col.reduce_scatter(bufs, 1.0 / K)
    sy = col.allgather_matmul(xd, wd)
    torch.cuda.synchronize()
    a, b = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    ev = torch.cuda.Event()
    ev.record()
    a.wait_event(ev)
    b.wait_event(ev)
    with torch.cuda.stream(b):
        c32, c16 = col.reduce_scatter(bufs, 1.0 / K, stream=b)
    with torch.cuda.stream(a):
        cy = col.allgather_matmul(xd, wd, stream=a)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    # the settle against the oracle: the ring fold of the sampled elements of
    # every rank (each sampled element is an 8-rank, one-element-per-chunk
    # problem placed at its own chunk index)
    rng = np.random.default_rng(31)
    idx = np.unique(np.concatenate([rng.integers(0, N, 2048), [0, C - 1, C, N - 1]]))
    it = torch.from_numpy(idx).to(DEV)
    host = [workloads.torch_bf16_to_bits(bf[it]) for bf in bufs]
    got32 = torch.cat(c32)[it].cpu().numpy().view(np.uint32)
    got16 = workloads.torch_bf16_to_bits(torch.cat(c16)[it])
    for q, e in enumerate(idx):
        c = int(e) // C
        col_in = [np.full(K, host[r][q], np.uint16) for r in range(K)]
        w32, w16 = oracle.reduce_scatter(col_in, 1.0 / K)
        assert got32[q] == w32[c].view(np.uint32)[0], (e, c)
        assert got16[q] == w16[c][0], (e, c)
    for c in range(K):
        assert torch.equal(ibits(c32[c]), ibits(s32[c]))
        assert torch.equal(ibits(c16[c]), ibits(s16[c]))
    # the GEMM against the fp64 oracle on sampled entries
    ms, fs = rng.integers(0, M, 600), rng.integers(0, 8 * Fs, 600)
    ref = oracle.allgather_matmul_f64_sampled(x, ws, ms, fs)
    val = cy.float().cpu().numpy()[ms, fs].astype(np.float64)
    assert np.linalg.norm(val - ref) / np.linalg.norm(ref) <= 1e-2
    assert torch.equal(ibits(cy), ibits(sy))


def _ag_inputs(K, C, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return [torch.randn(C, generator=g, device=DEV) for _ in range(K)]


def test_copy_engine_all_gather_on_a_side_stream_at_bench_size():
    # 8 shards x 16 MiB (the concurrency row's size); the copies run on the
    # library's internal streams and are joined back to the caller's stream
    K, C = 8, 16 * 1024 * 1024 // 4
    shards = _ag_inputs(K, C, 3)
    outs = [torch.full((K * C,), float("nan"), device=DEV) for _ in range(K)]
    side = torch.cuda.Stream(device=DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        B.dp_all_gather_copy_engine(shards, K, C, torch.float32, outs)
        # consumed on the same stream right away: ordered after the copies
        sums = torch.stack([o.view(torch.int32).sum(dtype=torch.int64) for o in outs])
    torch.cuda.current_stream().wait_stream(side)
    want = torch.cat(shards).view(torch.int32)
    for r in range(K):
        assert torch.equal(outs[r].view(torch.int32), want)
    assert torch.equal(sums, want.sum(dtype=torch.int64).repeat(K))


def test_copy_engine_all_gather_in_a_cuda_graph():
    K, C = 8, 3 * 4096
    shards = [torch.empty(C, device=DEV) for _ in range(K)]
    outs = [torch.empty(K * C, device=DEV) for _ in range(K)]
    side = torch.cuda.Stream(device=DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first call outside capture creates the streams
        B.dp_all_gather_copy_engine(shards, K, C, torch.float32, outs)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.dp_all_gather_copy_engine(shards, K, C, torch.float32, outs)
    for seed in (11, 12):
        for s, v in zip(shards, _ag_inputs(K, C, seed)):
            s.copy_(v)
        g.replay()
        torch.cuda.synchronize()
        want = torch.cat(shards).view(torch.int32)
        for r in range(K):
            assert torch.equal(outs[r].view(torch.int32), want)


def test_copy_engine_all_gather_from_two_host_threads():
    import threading
    K, C = 8, 1 << 20
    jobs = []
    for seed in (21, 22):
        shards = _ag_inputs(K, C, seed)
        outs = [torch.empty(K * C, device=DEV) for _ in range(K)]
        jobs.append((shards, outs, torch.cuda.Stream(device=DEV)))
    torch.cuda.synchronize()
    errs = []

    def work(shards, outs, st):
        try:
            for _ in range(5):
                assert B.dp_all_gather_copy_engine(shards, K, C, torch.float32, outs,
                                                   st.cuda_stream) == B.DP_OK
        except Exception as e:  # reported below
            errs.append(e)

    ts = [threading.Thread(target=work, args=j) for j in jobs]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    torch.cuda.synchronize()
    assert not errs
    for shards, outs, _ in jobs:
        want = torch.cat(shards).view(torch.int32)
        assert all(torch.equal(o.view(torch.int32), want) for o in outs)
