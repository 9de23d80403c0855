"""GPU parity of the ring collectives against the CPU oracle, bit for bit.

Sizes span many CTAs' worth of work plus ragged tails; misaligned views take
the scalar path; outputs sit between sentinel-filled guard regions that must
come back untouched.  Everything goes through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SENT32 = 0x7FC0DEAD  # a NaN pattern no kernel here writes
SENT16 = 0x7FCD
GUARD = 4096  # bytes on each side


def f32bits(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def bf16bits(t):
    return workloads.torch_bf16_to_bits(t)


def dev_tensor(a: np.ndarray):
    if a.dtype == np.uint16:
        return workloads.bits_to_torch_bf16(a).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Guarded:
    """n elements of dtype inside a larger buffer with sentinel guard bands;
    offset (elements) shifts the view off 16-byte alignment when non-zero."""

    def __init__(self, n, dtype, offset=0):
        esz = 4 if dtype == torch.float32 else 2
        g = GUARD // esz
        self.raw = torch.empty(2 * g + n + offset, dtype=torch.int32 if esz == 4 else torch.int16,
                               device=DEV)
        self.raw.fill_(SENT32 if esz == 4 else SENT16)
        self.g, self.n, self.off = g, n, offset
        self.t = self.raw[g + offset:g + offset + n].view(dtype)

    def guards_intact(self):
        lo = self.raw[:self.g + self.off].cpu()
        hi = self.raw[self.g + self.off + self.n:].cpu()
        s = SENT32 if self.raw.dtype == torch.int32 else SENT16
        return bool((lo == s).all()) and bool((hi == s).all())


def rand_ranks(K, N, dt, seed):
    rng = np.random.default_rng(seed)
    f = [rng.uniform(-1, 1, N).astype(np.float32) for _ in range(K)]
    return [workloads.to_bf16_bits(a) for a in f] if dt == "bf16" else f


# ---------------------------------------------------------------------------
# reduce-scatter
# ---------------------------------------------------------------------------

def test_config1_reduce_scatter_is_the_exact_sum():
    host = workloads.ring_ints(K=4, N=4096, seed=0)
    bufs = [dev_tensor(h) for h in host]
    o32, o16 = col.reduce_scatter(bufs, 1.0)
    exact = np.sum(np.stack(host).astype(np.int64), axis=0).astype(np.float32)
    r32, r16 = oracle.reduce_scatter(host, 1.0)
    for c in range(4):
        assert np.array_equal(f32bits(o32[c]), exact[c * 1024:(c + 1) * 1024].view(np.uint32))
        assert np.array_equal(f32bits(o32[c]), r32[c].view(np.uint32))
        assert np.array_equal(bf16bits(o16[c]), r16[c])


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 8, 11, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_reduce_scatter_matches_oracle(K, dt):
    C = 8 * 2053  # many CTA strides of 8-element units, odd unit count
    N = K * C
    host = rand_ranks(K, N, dt, 17 * K)
    bufs = [dev_tensor(h) for h in host]
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    g32 = [Guarded(C, torch.float32) for _ in range(K)]
    g16 = [Guarded(C, torch.bfloat16) for _ in range(K)]
    scale = 1.0 / K
    B.dp_reduce_scatter_dual(bufs, K, N, tdt, [g.t for g in g32], [g.t for g in g16], scale)
    torch.cuda.synchronize()
    r32, r16 = oracle.reduce_scatter(host, scale)
    for c in range(K):
        assert np.array_equal(f32bits(g32[c].t), r32[c].view(np.uint32)), c
        assert np.array_equal(bf16bits(g16[c].t), r16[c]), c
        assert g32[c].guards_intact() and g16[c].guards_intact()


@pytest.mark.parametrize("K,C,off_in,off_out", [(4, 1003, 0, 0), (8, 8 * 100, 1, 0),
                                                (8, 8 * 100, 0, 1), (3, 5, 0, 0),
                                                (16, 1, 0, 0)])
def test_reduce_scatter_scalar_path(K, C, off_in, off_out):
    N = K * C
    host = rand_ranks(K, N, "bf16", K + C)
    ins = [Guarded(N, torch.bfloat16, off_in) for _ in range(K)]
    for g, h in zip(ins, host):
        g.t.copy_(workloads.bits_to_torch_bf16(h))
    outs = [Guarded(C, torch.float32, off_out) for _ in range(K)]
    B.dp_reduce_scatter([g.t for g in ins], K, N, B.DP_BF16, [g.t for g in outs], 0.3, B.DP_FP32)
    torch.cuda.synchronize()
    r32, _ = oracle.reduce_scatter(host, 0.3, ("f32",))
    for c in range(K):
        assert np.array_equal(f32bits(outs[c].t), r32[c].view(np.uint32))
        assert outs[c].guards_intact()


def test_reduce_scatter_single_output_types():
    K, N = 8, 8 * 4096
    host = rand_ranks(K, N, "f32", 3)
    bufs = [dev_tensor(h) for h in host]
    o16 = [torch.empty(N // K, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    B.dp_reduce_scatter(bufs, K, N, B.DP_FP32, o16, 0.125, B.DP_BF16)
    o32, _ = col.reduce_scatter(bufs, 0.125, ("f32",))
    r32, r16 = oracle.reduce_scatter(host, 0.125)
    for c in range(K):
        assert np.array_equal(bf16bits(o16[c]), r16[c])
        assert np.array_equal(f32bits(o32[c]), r32[c].view(np.uint32))


def test_reduce_scatter_full_fsdp_gradient_sampled():
    """K=8 ranks of 64 Mi bf16 gradients, fp32 + bf16 shards, scale 1/8 --
    the full-size workload in the benchmark's launch configuration, checked
    on sampled elements against the oracle and everywhere by the property
    bf16 shard == RNE(fp32 shard)."""
    K, N = 8, 64 * workloads.MiB
    C = N // K
    bufs = workloads.fsdp_grads_device(K, N, DEV)
    o32, o16 = col.reduce_scatter(bufs, 1.0 / K)
    torch.cuda.synchronize()
    rng = np.random.default_rng(99)
    idx = np.unique(np.concatenate([rng.integers(0, N, 4096), [0, C - 1, C, N - 1]]))
    S = idx.size
    vals = torch.stack([b[torch.from_numpy(idx).to(DEV)] for b in bufs]).cpu()
    vals = vals.view(torch.int16).numpy().view(np.uint16)  # [K, S] bf16 bits
    # one small oracle problem: sample s of chunk c sits at position c*S + s
    small = [np.zeros(K * S, np.uint16) for _ in range(K)]
    chunk = idx // C
    for r in range(K):
        small[r][chunk * S + np.arange(S)] = vals[r]
    r32, r16 = oracle.reduce_scatter(small, 1.0 / K)
    got32 = np.stack([f32bits(o32[c]) for c in range(K)])
    got16 = np.stack([bf16bits(o16[c]) for c in range(K)])
    for s, e in enumerate(idx):
        c, i = divmod(int(e), C)
        assert got32[c, i] == r32[c][s].view(np.uint32), e
        assert got16[c, i] == r16[c][s], e
    for c in range(K):
        assert torch.equal(o32[c].to(torch.bfloat16).view(torch.int16), o16[c].view(torch.int16))


# ---------------------------------------------------------------------------
# all-gather
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 2, 4, 7, 8, 16])
@pytest.mark.parametrize("dt,C,off", [("f32", 4 * 3001, 0), ("bf16", 8 * 3001, 0),
                                      ("bf16", 1001, 0), ("f32", 64, 1),
                                      ("f32", 4 * 3001 + 16384 * 2, 4), ("bf16", 8 * 3001, 8)])
def test_all_gather_matches_oracle(K, dt, C, off):
    """Offsets of 4 f32 / 8 bf16 elements keep the views 16-byte aligned (the
    bulk-copy path) but off every larger boundary; offset 1 takes the scalar
    path.  Guard bands around every output catch a stray write."""
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    host = rand_ranks(K, C, dt, 5 * K + C)
    shards = [Guarded(C, tdt, off) for _ in range(K)]
    for g, h in zip(shards, host):
        g.t.copy_(dev_tensor(h))
    outs = [Guarded(K * C, tdt, off) for _ in range(K)]
    B.dp_all_gather([g.t for g in shards], K, C, tdt, [g.t for g in outs])
    torch.cuda.synchronize()
    ref = oracle.all_gather(host)
    for r in range(K):
        got = f32bits(outs[r].t) if dt == "f32" else bf16bits(outs[r].t)
        want = ref[r].view(np.uint32) if dt == "f32" else ref[r]
        assert np.array_equal(got, want)
        assert outs[r].guards_intact()


# ---------------------------------------------------------------------------
# all-reduce
# ---------------------------------------------------------------------------

def test_config1_allreduce_every_rank_holds_the_sum():
    host = workloads.ring_ints(K=4, N=4096, seed=0)
    bufs = [dev_tensor(h) for h in host]
    col.all_reduce_(bufs, 1.0)
    exact = np.sum(np.stack(host).astype(np.int64), axis=0).astype(np.float32)
    for r in range(4):
        assert np.array_equal(f32bits(bufs[r]), exact.view(np.uint32))


@pytest.mark.parametrize("K", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N", [8 * 5 * 1024, 8 * 5 * 1024 + 3, 999, 5])
def test_allreduce_matches_oracle(K, dt, N):
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    host = rand_ranks(K, N, dt, 31 * K + N)
    bufs = [Guarded(N, tdt) for _ in range(K)]
    for g, h in zip(bufs, host):
        g.t.copy_(dev_tensor(h))
    B.dp_ring_allreduce([g.t for g in bufs], K, N, tdt, 1.0 / K)
    torch.cuda.synchronize()
    ref = oracle.all_reduce(host, 1.0 / K)
    for r in range(K):
        got = f32bits(bufs[r].t) if dt == "f32" else bf16bits(bufs[r].t)
        want = ref[r].view(np.uint32) if dt == "f32" else ref[r]
        assert np.array_equal(got, want)
        assert bufs[r].guards_intact()


def test_allreduce_short_last_chunk_vector_path():
    # C = ceil(N/K) is a multiple of 8, the last chunk is short and ragged
    K, N = 8, 8 * 8 * 1000 - 13
    host = rand_ranks(K, N, "f32", 77)
    bufs = [dev_tensor(h) for h in host]
    col.all_reduce_(bufs, 0.125)
    ref = oracle.all_reduce(host, 0.125)
    for r in range(K):
        assert np.array_equal(f32bits(bufs[r]), ref[r].view(np.uint32))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_allreduce_equals_reduce_scatter_then_all_gather(dt):
    K, N = 8, 8 * 8 * 777
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    host = rand_ranks(K, N, dt, 8)
    a = [dev_tensor(h) for h in host]
    b = [x.clone() for x in a]
    col.all_reduce_(a, 1.0 / K)
    o32, o16 = col.reduce_scatter(b, 1.0 / K)
    shards = o32 if dt == "f32" else o16
    g = col.all_gather(shards)
    for r in range(K):
        assert torch.equal(a[r].view(torch.int16 if dt == "bf16" else torch.int32),
                           g[r].view(torch.int16 if dt == "bf16" else torch.int32))
        assert torch.equal(a[r].view(torch.uint8), a[0].view(torch.uint8))


@pytest.mark.parametrize("K", [2, 4, 8])
def test_sweep_sizes_small_match_oracle(K):
    # the bandwidth sweep's per-rank sizes 4 KiB .. 4 MiB in full
    for nbytes in workloads.sweep_sizes_bytes()[:6]:
        N = nbytes // 4
        host = workloads.sweep_bufs(K, N)
        bufs = [dev_tensor(h) for h in host]
        col.all_reduce_(bufs, 1.0 / K)
        ref = oracle.all_reduce(host, 1.0 / K)
        for r in range(K):
            assert np.array_equal(f32bits(bufs[r]), ref[r].view(np.uint32)), (K, nbytes, r)


@pytest.mark.parametrize("K", [2, 4, 8])
def test_sweep_largest_size_sampled(K):
    """K x 1 GiB fp32 per rank, in place: sampled elements vs the oracle."""
    N = (1 << 30) // 4
    C = N // K
    bufs = workloads.sweep_bufs_device(K, N, DEV)
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, N, 2048), [0, C - 1, C, N - 1]]))
    it = torch.from_numpy(idx).to(DEV)
    vals = torch.stack([b[it] for b in bufs]).cpu().numpy()
    col.all_reduce_(bufs, 1.0 / K)
    torch.cuda.synchronize()
    S = idx.size
    small = [np.zeros(K * S, np.float32) for _ in range(K)]
    for r in range(K):
        small[r][(idx // C) * S + np.arange(S)] = vals[r]
    r32, _ = oracle.reduce_scatter(small, 1.0 / K, ("f32",))
    for r in sorted({0, K // 2, K - 1}):
        got = bufs[r][it].cpu().numpy().view(np.uint32)
        want = np.array([r32[int(e) // C][s] for s, e in enumerate(idx)], np.float32)
        assert np.array_equal(got, want.view(np.uint32))
    del bufs
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# errors, device error word
# ---------------------------------------------------------------------------

def test_alias_is_rejected_with_real_buffers():
    x = torch.zeros(4096, device=DEV)
    views = [x[0:1024], x[512:1536], x[2048:3072], x[3072:4096]]
    assert B.dp_ring_allreduce(views, 4, 1024, B.DP_FP32, 1.0, check=False) == B.DP_ERR_ALIAS
    assert B.dp_get_device_error() == B.DP_OK


def test_bounded_wait_expiry_is_reported_and_cleared():
    assert B.dp_get_device_error() == B.DP_OK
    B.dp_selftest_bounded_wait(2000)  # 2 ms on a barrier nothing completes
    assert B.dp_get_device_error() == B.DP_ERR_TIMEOUT
    assert B.dp_get_device_error() == B.DP_OK
    # the context is still usable afterwards
    host = workloads.ring_ints(K=4, N=64, seed=2)
    bufs = [dev_tensor(h) for h in host]
    col.all_reduce_(bufs, 1.0)
    exact = np.sum(np.stack(host), axis=0).astype(np.float32)
    assert np.array_equal(bufs[1].cpu().numpy(), exact)


def test_reduce_scatter_reads_and_writes_pinned_host_buffers():
    """Zero-copy: the same call on pinned host inputs and outputs gives the
    same bits as on device buffers."""
    K, N = 8, 8 * 8 * 4099
    dev_in = workloads.fsdp_grads_device(K, N, DEV)
    host_in = [t.cpu().pin_memory() for t in dev_in]
    C = N // K
    h32 = [torch.empty(C, dtype=torch.float32).pin_memory() for _ in range(K)]
    h16 = [torch.empty(C, dtype=torch.bfloat16).pin_memory() for _ in range(K)]
    B.dp_reduce_scatter_dual(host_in, K, N, B.DP_BF16, h32, h16, 1.0 / K)
    d32, d16 = col.reduce_scatter(dev_in, 1.0 / K)
    torch.cuda.synchronize()
    for c in range(K):
        assert torch.equal(h32[c].view(torch.int32), d32[c].cpu().view(torch.int32))
        assert torch.equal(h16[c].view(torch.int16), d16[c].cpu().view(torch.int16))


@pytest.mark.parametrize("scale", [0.0, -1.0, 1e-40, 3.0e38, -0.125])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_degenerate_scales_match_oracle(scale, dt):
    """Signed zeros (scale 0 keeps the fold's sign), negative scales, fp32
    denormals (no flush to zero) and overflow to +-inf, bit for bit, in the
    reduce-scatter (both outputs) and the all-reduce (both variants)."""
    K, N = 8, 8 * 8 * 513
    host = rand_ranks(K, N, dt, 123)
    bufs = [dev_tensor(h) for h in host]
    o32, o16 = col.reduce_scatter(bufs, scale)
    r32, r16 = oracle.reduce_scatter(host, scale)
    for c in range(K):
        assert np.array_equal(f32bits(o32[c]), r32[c].view(np.uint32))
        assert np.array_equal(bf16bits(o16[c]), r16[c])
    ref = oracle.all_reduce(host, scale)
    for variant in (1, 2):
        B.dp_set_collective_variant(variant)
        try:
            ar = [dev_tensor(h) for h in host]
            col.all_reduce_(ar, scale)
            torch.cuda.synchronize()
        finally:
            B.dp_set_collective_variant(0)
        for r in range(K):
            got = f32bits(ar[r]) if dt == "f32" else bf16bits(ar[r])
            want = ref[r].view(np.uint32) if dt == "f32" else ref[r]
            assert np.array_equal(got, want), (variant, r)


# ---------------------------------------------------------------------------
# CUDA graphs: every call only enqueues kernels with by-value parameters, so
# a captured sequence replays on whatever the buffers hold at replay time
# ---------------------------------------------------------------------------

def test_collectives_captured_in_a_cuda_graph_replay_on_new_inputs():
    K, C = 4, 8 * 1501
    N = K * C
    rs_in = [torch.empty(N, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    o32 = [torch.empty(C, device=DEV) for _ in range(K)]
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    ag_out = [torch.empty(N, device=DEV) for _ in range(K)]
    ar_buf = [torch.empty(N + 5, device=DEV) for _ in range(K)]  # ragged all-reduce
    m = [2, 0, 3, 1]
    odc_g = [[torch.empty(N, dtype=torch.bfloat16, device=DEV) for _ in range(m[r])]
             for r in range(K)]

    def sequence():
        B.dp_reduce_scatter_dual(rs_in, K, N, torch.bfloat16, o32, o16, 1.0 / K)
        B.dp_all_gather(o32, K, C, torch.float32, ag_out)
        B.dp_ring_allreduce(ar_buf, K, N + 5, torch.float32, 0.5)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # once eagerly: kernel attributes are set outside capture
        sequence()
        col.odc_reduce_scatter(odc_g, m, N, 1.0 / K)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sequence()
        og32, og16 = col.odc_reduce_scatter(odc_g, m, N, 1.0 / K)
    for seed in (21, 22):
        rng = np.random.default_rng(seed)
        h_rs = [workloads.to_bf16_bits(rng.uniform(-1, 1, N).astype(np.float32)) for _ in range(K)]
        h_ar = [rng.uniform(-1, 1, N + 5).astype(np.float32) for _ in range(K)]
        h_odc = [[workloads.to_bf16_bits(rng.standard_normal(N).astype(np.float32) *
                                         np.float32(1e-3)) for _ in range(m[r])] for r in range(K)]
        for t, h in zip(rs_in, h_rs):
            t.copy_(dev_tensor(h))
        for t, h in zip(ar_buf, h_ar):
            t.copy_(dev_tensor(h))
        for r in range(K):
            for t, h in zip(odc_g[r], h_odc[r]):
                t.copy_(dev_tensor(h))
        g.replay()
        torch.cuda.synchronize()
        assert B.dp_get_device_error() == B.DP_OK
        r32, r16 = oracle.reduce_scatter(h_rs, 1.0 / K)
        ref_ag = oracle.all_gather(r32)
        ref_ar = oracle.all_reduce(h_ar, 0.5)
        e32, e16 = oracle.odc_layer(h_odc, m, 1.0 / K, N)
        for c in range(K):
            assert np.array_equal(f32bits(o32[c]), r32[c].view(np.uint32)), (seed, c)
            assert np.array_equal(bf16bits(o16[c]), r16[c]), (seed, c)
            assert np.array_equal(f32bits(ag_out[c]), ref_ag[c].view(np.uint32)), (seed, c)
            assert np.array_equal(f32bits(ar_buf[c]), ref_ar[c].view(np.uint32)), (seed, c)
            assert np.array_equal(f32bits(og32[c]), e32[c].view(np.uint32)), (seed, c)
            assert np.array_equal(bf16bits(og16[c]), e16[c]), (seed, c)
