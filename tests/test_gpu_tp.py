"""GPU parity of the tensor-parallel psum fused into the GEMM
(dp_matmul_allreduce / dp_matmul_reduce_scatter) against the fp64 oracle.

Bar: normwise relative error <= 1e-2 (fp32 accumulation order is the tensor
core's); integer operands give exact results; every rank's all-reduce output
is bitwise identical, and the reduce-scatter shards are bitwise the matching
rows of the all-reduce result.
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
TOL = 1e-2


def to_dev(bits):
    return workloads.bits_to_torch_bf16(bits).to(DEV)


def rel_err(y, ref):
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
def test_tp_fixture_1024x64x512_k8(ydt):
    """The TP-style fixture: x_r[1024, 64] and a 512-wide partial per rank,
    summed eight ways."""
    K, M, Ds, F = 8, 1024, 64, 512
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    xd, wd = [to_dev(x) for x in xs], [to_dev(w) for w in ws]
    ys = col.matmul_allreduce(xd, wd, 1.0, ydt)
    shards = col.matmul_reduce_scatter(xd, wd, 1.0, ydt)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    ref = oracle.matmul_psum_f64(xs, ws)
    y0 = ys[0].double().cpu().numpy()
    assert rel_err(y0, ref) <= TOL
    iv = torch.int16 if ydt == torch.bfloat16 else torch.int32
    for r in range(1, K):
        assert torch.equal(ys[r].view(iv), ys[0].view(iv))
    rows = M // K
    for c in range(K):
        assert torch.equal(shards[c].view(iv), ys[0][c * rows:(c + 1) * rows].view(iv))


@pytest.mark.parametrize("K,M,Ds,F", [(8, 256, 64, 128), (4, 512, 128, 256), (2, 128, 512, 64)])
def test_tp_integer_operands_exact(K, M, Ds, F):
    xs, ws = workloads.tp_operands(M, Ds, F, K, ints=True)
    ys = col.matmul_allreduce([to_dev(x) for x in xs], [to_dev(w) for w in ws], 1.0,
                              torch.float32)
    ref = oracle.matmul_psum_f64(xs, ws)
    assert np.array_equal(ys[K - 1].double().cpu().numpy(), ref)


@pytest.mark.parametrize("K,M,Ds,F,scale", [(8, 200, 72, 96, 1.0), (3, 384, 40, 48, 0.5),
                                            (16, 128, 16, 32, 1.0 / 16), (1, 300, 256, 512, 1.0)])
def test_tp_shapes_allreduce(K, M, Ds, F, scale):
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    ys = col.matmul_allreduce([to_dev(x) for x in xs], [to_dev(w) for w in ws], scale,
                              torch.float32)
    ref = oracle.matmul_psum_f64(xs, ws, scale)
    assert rel_err(ys[0].double().cpu().numpy(), ref) <= TOL


def test_tp_full_size_reduce_scatter_sampled():
    K, M, Ds, F = 8, 8192, 512, 4096
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    shards = col.matmul_reduce_scatter([to_dev(x) for x in xs], [to_dev(w) for w in ws], 1.0,
                                       torch.bfloat16)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    rng = np.random.default_rng(3)
    ms = np.concatenate([rng.integers(0, M, 1000), [0, M - 1, M // K - 1, M // K]])
    fs = np.concatenate([rng.integers(0, F, 1000), [0, F - 1, 255, 256]])
    ref = oracle.matmul_psum_f64_sampled(xs, ws, ms, fs)
    rows = M // K
    got = np.array([float(shards[m // rows][m % rows, f]) for m, f in zip(ms, fs)])
    assert rel_err(got, ref) <= TOL


def test_tp_reduce_scatter_rejects_uneven_rows():
    xs = [torch.zeros(100, 64, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    ws = [torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    ys = [torch.zeros(12, 64, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    st = B.dp_matmul_reduce_scatter(xs, ws, 8, 100, 64, 64, ys, B.DP_BF16, 1.0, check=False)
    assert st == B.DP_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# The x . w orientation of the page's fixture ("Sharding and Parallelism",
# "Real HLO before and after partitioning": x[1024,64] @ w[64,512] per rank,
# w sharded along its contracted rows): w_r given [D_shard, F] row-major.
# ---------------------------------------------------------------------------

def _kn(ws):
    """The same weights in the [D_shard, F] layout (numpy transpose)."""
    return [np.ascontiguousarray(w.T) for w in ws]


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
def test_tp_xw_fixture_1024x64_at_64x512_k8(ydt):
    K, M, Ds, F = 8, 1024, 64, 512
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    xd = [to_dev(x) for x in xs]
    wkn = [to_dev(w) for w in _kn(ws)]
    ys = col.matmul_allreduce_xw(xd, wkn, 1.0, ydt)
    shards = col.matmul_reduce_scatter_xw(xd, wkn, 1.0, ydt)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    ref = oracle.matmul_psum_f64(xs, ws)
    assert rel_err(ys[0].double().cpu().numpy(), ref) <= TOL
    iv = torch.int16 if ydt == torch.bfloat16 else torch.int32
    rows = M // K
    for r in range(K):
        assert torch.equal(ys[r].view(iv), ys[0].view(iv))
        assert torch.equal(shards[r].view(iv), ys[0][r * rows:(r + 1) * rows].view(iv))
    # the same products in the same k order as the [F, D_shard] form: the
    # tensor core's sums do not depend on how its operands sit in shared memory
    yk = col.matmul_allreduce(xd, [to_dev(w) for w in ws], 1.0, ydt)
    assert torch.equal(ys[0].view(iv), yk[0].view(iv))


@pytest.mark.parametrize("K,M,Ds,F", [(8, 256, 64, 128), (4, 512, 128, 256), (2, 128, 512, 64)])
def test_tp_xw_integer_operands_exact(K, M, Ds, F):
    xs, ws = workloads.tp_operands(M, Ds, F, K, ints=True)
    ys = col.matmul_allreduce_xw([to_dev(x) for x in xs], [to_dev(w) for w in _kn(ws)], 1.0,
                                 torch.float32)
    ref = oracle.matmul_psum_f64(xs, ws)
    assert np.array_equal(ys[K - 1].double().cpu().numpy(), ref)


@pytest.mark.parametrize("K,M,Ds,F,scale", [(8, 200, 72, 128, 1.0), (3, 384, 40, 64, 0.5),
                                            (16, 128, 16, 64, 1.0 / 16), (1, 300, 256, 512, 1.0),
                                            (8, 1000, 96, 192, 0.125)])
def test_tp_xw_shapes(K, M, Ds, F, scale):
    """Ragged rows, contracted lengths that are not a whole k-block (the
    tail of the last block of w_r's rows is read as zeros), narrow tiles."""
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    xd, wkn = [to_dev(x) for x in xs], [to_dev(w) for w in _kn(ws)]
    ys = col.matmul_allreduce_xw(xd, wkn, scale, torch.float32)
    ref = oracle.matmul_psum_f64(xs, ws, scale)
    assert rel_err(ys[0].double().cpu().numpy(), ref) <= TOL
    if M % K == 0:
        shards = col.matmul_reduce_scatter_xw(xd, wkn, scale, torch.float32)
        rows = M // K
        for c in range(K):
            assert torch.equal(shards[c].view(torch.int32),
                               ys[0][c * rows:(c + 1) * rows].view(torch.int32))


def test_tp_xw_full_size_reduce_scatter_sampled():
    K, M, Ds, F = 8, 8192, 512, 4096
    xs, ws = workloads.tp_operands(M, Ds, F, K)
    shards = col.matmul_reduce_scatter_xw([to_dev(x) for x in xs], [to_dev(w) for w in _kn(ws)],
                                          1.0, torch.bfloat16)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    rng = np.random.default_rng(5)
    ms = np.concatenate([rng.integers(0, M, 1000), [0, M - 1, M // K - 1, M // K]])
    fs = np.concatenate([rng.integers(0, F, 1000), [0, F - 1, 255, 256]])
    ref = oracle.matmul_psum_f64_sampled(xs, ws, ms, fs)
    rows = M // K
    got = np.array([float(shards[m // rows][m % rows, f]) for m, f in zip(ms, fs)])
    assert rel_err(got, ref) <= TOL


def test_tp_xw_rejects_a_width_that_is_not_whole_slabs():
    xs = [torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    ws = [torch.zeros(64, 96, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    ys = [torch.full((128, 96), 3.0, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    st = B.dp_matmul_allreduce_xw(xs, ws, 2, 128, 64, 96, ys, B.DP_BF16, 1.0, check=False)
    assert st == B.DP_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert all(bool((y == 3.0).all()) for y in ys)


@pytest.mark.parametrize("K,M,Ds,F", [(16, 256, 8, 64), (16, 640, 128, 320)])
def test_tp_xw_sixteen_ranks_and_short_rows(K, M, Ds, F):
    """Sixteen ranks, and the shortest contracted length (8: one 16-byte row
    of x_r, w_r's slabs mostly zero fill); integer operands are exact."""
    xs, ws = workloads.tp_operands(M, Ds, F, K, ints=True)
    xd, wkn = [to_dev(x) for x in xs], [to_dev(w) for w in _kn(ws)]
    ys = col.matmul_allreduce_xw(xd, wkn, 1.0, torch.float32)
    ref = oracle.matmul_psum_f64(xs, ws)
    assert np.array_equal(ys[K - 1].double().cpu().numpy(), ref)
    shards = col.matmul_reduce_scatter_xw(xd, wkn, 1.0, torch.float32)
    rows = M // K
    for c in range(K):
        assert torch.equal(shards[c].view(torch.int32),
                           ys[0][c * rows:(c + 1) * rows].view(torch.int32))


def test_degenerate_gemm_shapes():
    """An empty contraction (D = 0, D_shard = 0) writes zeros to every
    output; an empty output (M = 0) touches nothing."""
    K = 8
    x = torch.ones(128, 8, dtype=torch.bfloat16, device=DEV)
    ws = [torch.ones(64, 8, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    y = torch.full((128, 512), 7.0, device=DEV)
    B.dp_allgather_matmul(x, 128, 0, ws, K, 64, y, B.DP_FP32)
    torch.cuda.synchronize()
    assert bool((y == 0).all())
    y.fill_(7.0)
    B.dp_allgather_matmul(x, 0, 8, ws, K, 64, y, B.DP_FP32)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    xs = [torch.ones(64, 8, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    wt = [torch.ones(32, 8, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    ys = [torch.full((64, 32), 7.0, device=DEV) for _ in range(K)]
    B.dp_matmul_allreduce(xs, wt, K, 64, 0, 32, ys, B.DP_FP32, 1.0)
    shards = [torch.full((8, 32), 7.0, device=DEV) for _ in range(K)]
    B.dp_matmul_reduce_scatter(xs, wt, K, 64, 0, 32, shards, B.DP_FP32, 1.0)
    torch.cuda.synchronize()
    assert all(bool((t == 0).all()) for t in ys + shards)
    for t in ys:
        t.fill_(7.0)
    B.dp_matmul_allreduce(xs, wt, K, 0, 8, 32, ys, B.DP_FP32, 1.0)
    torch.cuda.synchronize()
    assert all(bool((t == 7.0).all()) for t in ys)
    assert B.dp_get_device_error() == B.DP_OK
