"""GPU parity: the chained split of a part-full last round in the gather GEMM
and the tensor-parallel GEMMs.

With a workspace, the tiles left over after the persistent grid's whole
rounds (at most half a round) are cut into k-block segments on different
CTAs, each continuing the previous one's fp32 accumulator, so every output
element sees the same MMAs in the same order and the result must be bitwise
the one without the split (and the same under any CTA limit).  CTA limits
make small problems split into 2, 3 and 4 segments; larger shapes split at
the GPU's own CTA count.
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
TOL = 1e-2


def plan(tiles, grid, num_kb, bn, max_split=4, min_seg_kb=8):
    """The split the library is expected to choose: (segments, workspace
    bytes), or None.  Only a last round at most half full is split, into as
    many segments as fit on the idle CTAs (one each), at most 4, at most
    q + 1, each >= 8 k-blocks."""
    q, R = divmod(tiles, grid)
    if grid < 2 or q < 1 or R == 0 or 2 * R > grid:
        return None
    s = min(grid // R, q + 1, max_split)
    while s > 1 and num_kb // s < min_seg_kb:
        s -= 1
    if s < 2:
        return None
    parts = (s - 1) * R
    return s, (parts * 8 + 255) // 256 * 256 + parts * 128 * bn * 4


@pytest.fixture
def cta_limit():
    saved = B.dp_get_cta_limits()

    def set_gemm(n):
        B.dp_set_cta_limits(n, 0)

    yield set_gemm
    B.dp_set_cta_limits(*saved)


def _bits(ts):
    return [t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32) for t in ts]


def _equal(a, b):
    return all(torch.equal(p, q) for p, q in zip(_bits(a), _bits(b)))


# (CTA limit, M, D, F_shard, expected segments): 128 tiles of 128 x 64 (the
# width the library picks for M = 2048, F = 512: a problem with fewer tiles
# than half the SMs' count gets narrower ones)
GATHER = [(63, 2048, 2048, 64, 3), (41, 2048, 2048, 64, 4), (100, 2048, 1024, 64, 2)]


@pytest.mark.parametrize("limit,M,D,Fs,segs", GATHER)
def test_gather_gemm_split_is_bitwise_the_unsplit_result(cta_limit, limit, M, D, Fs, segs):
    K = 8
    x, ws = workloads.gemm_operands(M, D, K, Fs)
    xd = workloads.bits_to_torch_bf16(x).to(DEV)
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    cta_limit(limit)
    need = B.dp_allgather_matmul_workspace_size(M, D, K, Fs)
    tiles, bn = (M // 128) * (K * Fs // 64), 64
    assert plan(tiles, limit, D // 64, bn) == (segs, need)
    plain = col.allgather_matmul(xd, wd, torch.float32, workspace=None)
    split = col.allgather_matmul(xd, wd, torch.float32)
    again = col.allgather_matmul(xd, wd, torch.float32)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    assert _equal([plain], [split]) and _equal([plain], [again])
    cta_limit(0)
    assert _equal([plain], [col.allgather_matmul(xd, wd, torch.float32, workspace=None)])
    rng = np.random.default_rng(limit)
    ms, fs = rng.integers(0, M, 2000), rng.integers(0, K * Fs, 2000)
    ref = oracle.allgather_matmul_f64_sampled(x, ws, ms, fs)
    got = split.double().cpu().numpy()[ms, fs]
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= TOL


# (CTA limit, M, D_shard, F, expected segments): 64 tiles of 128 x 64
TP = [(15, 1024, 256, 512, 3), (20, 1024, 256, 512, 4), (10, 1024, 128, 512, 2)]


@pytest.mark.parametrize("scatter", [False, True])
@pytest.mark.parametrize("limit,M,Ds,F,segs", TP)
def test_tp_gemm_split_is_bitwise_the_unsplit_result(cta_limit, scatter, limit, M, Ds, F, segs):
    K = 8
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    xd = [workloads.bits_to_torch_bf16(a).to(DEV) for a in xs]
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    fn = col.matmul_reduce_scatter if scatter else col.matmul_allreduce
    cta_limit(limit)
    need = B.dp_matmul_workspace_size(K, M, Ds, F)
    tiles, bn, num_kb = (M // 128) * (F // 64), 64, K * Ds // 64
    assert plan(tiles, limit, num_kb, bn) == (segs, need)
    plain = fn(xd, wd, 0.5, torch.bfloat16, workspace=None)
    split = fn(xd, wd, 0.5, torch.bfloat16)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    assert _equal(plain, split)
    rng = np.random.default_rng(limit)
    ms, fs = rng.integers(0, M, 2000), rng.integers(0, F, 2000)
    ref = oracle.matmul_psum_f64_sampled(xs, ws, ms, fs, 0.5)
    full = torch.cat(split, 0) if scatter else split[0]
    got = full.double().cpu().numpy()[ms, fs]
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= TOL


def test_split_tp_gemm_in_a_cuda_graph(cta_limit):
    # replays reuse the launch's flag value; each flag is cleared once read
    K, M, Ds, F = 8, 1024, 256, 512
    cta_limit(15)
    need = B.dp_matmul_workspace_size(K, M, Ds, F)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    xs = [torch.empty(M, Ds, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    wts = [torch.empty(F, Ds, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    ys = [torch.empty(M // K, F, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        B.dp_matmul_reduce_scatter(xs, wts, K, M, Ds, F, ys, B.DP_BF16, 1.0, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.dp_matmul_reduce_scatter(xs, wts, K, M, Ds, F, ys, B.DP_BF16, 1.0, workspace=ws)
    for seed in (1, 2, 3):
        gen = torch.Generator(device=DEV)
        gen.manual_seed(seed)
        for t in xs + wts:
            t.copy_((torch.randn(t.shape, generator=gen, device=DEV) * 0.05).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert B.dp_get_device_error() == B.DP_OK
        want = col.matmul_reduce_scatter(xs, wts, 1.0, torch.bfloat16, workspace=None)
        assert _equal(ys, want)


def test_large_shapes_split_is_bitwise_the_unsplit_result(cta_limit):
    """At the GPU's own CTA count: the gather GEMM x[4096,4096] . (8 shards
    [512,4096])^T and the TP GEMMs 8 x (x_r[5120,512] . w_r[4096,512]^T)
    (512 and 640 tiles of 128 x 256: 56 and 32 left over on 152 SMs).  The
    benchmark's M = 8192 shapes leave 112 of 152 and are not split."""
    cta_limit(0)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    K = 8
    g = torch.Generator(device=DEV)
    g.manual_seed(40)
    x = (torch.randn(4096, 4096, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w = [(torch.randn(512, 4096, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
         for _ in range(K)]
    p = plan(512, n_sm, 64, 256)
    assert B.dp_allgather_matmul_workspace_size(4096, 4096, K, 512) == (p[1] if p else 0)
    assert B.dp_allgather_matmul_workspace_size(8192, 4096, K, 512) == \
        (plan(1024, n_sm, 64, 256) or (0, 0))[1]
    if n_sm == 152:
        assert p[0] == 2
    assert _equal([col.allgather_matmul(x, w, workspace=None)], [col.allgather_matmul(x, w)])
    xs = [(torch.randn(5120, 512, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
          for _ in range(K)]
    ws = [(torch.randn(4096, 512, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
          for _ in range(K)]
    p = plan(640, n_sm, 64, 256)
    assert B.dp_matmul_workspace_size(K, 5120, 512, 4096) == (p[1] if p else 0)
    if n_sm == 152:
        assert p[0] == 4
    for fn in (col.matmul_allreduce, col.matmul_reduce_scatter):
        assert _equal(fn(xs, ws, 1.0, torch.bfloat16, workspace=None),
                      fn(xs, ws, 1.0, torch.bfloat16))
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK


def test_tp_split_with_fp32_output(cta_limit):
    K, M, Ds, F = 8, 1024, 256, 512
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    xd = [workloads.bits_to_torch_bf16(a).to(DEV) for a in xs]
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    cta_limit(20)
    assert B.dp_matmul_workspace_size(K, M, Ds, F) > 0
    for fn in (col.matmul_allreduce, col.matmul_reduce_scatter):
        plain = fn(xd, wd, 0.125, torch.float32, workspace=None)
        split = fn(xd, wd, 0.125, torch.float32)
        torch.cuda.synchronize()
        assert _equal(plain, split)


def test_tp_split_with_integer_operands_is_exact(cta_limit):
    # |values| <= 4, 8 ranks x 256 = 2048 products of <= 16 per output: every
    # partial sum is an integer below 2^24, exact in any order
    K, M, Ds, F = 8, 1024, 256, 512
    xs, ws = workloads.tp_operands(M, Ds, F, K, ints=True)
    xd = [workloads.bits_to_torch_bf16(a).to(DEV) for a in xs]
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    cta_limit(15)
    assert B.dp_matmul_workspace_size(K, M, Ds, F) > 0
    got = col.matmul_reduce_scatter(xd, wd, 1.0, torch.float32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    ms, fs = rng.integers(0, M, 3000), rng.integers(0, F, 3000)
    ref = oracle.matmul_psum_f64_sampled(xs, ws, ms, fs)
    full = torch.cat(got, 0).double().cpu().numpy()
    assert np.array_equal(full[ms, fs], ref)
