"""GPU parity: the FSDP backward weight gradient fused with its reduce-scatter.

"Using ODC to Accelerate AMD SFT Training", section "Why FSDP is Slow": each
layer's full gradient is computed in the backward pass and reduce-scattered to
the rank's shard.  Rank r's dW_r = dy_r^T x_r (tokens contracted); the fused
kernel chains every rank's token blocks into one fp32 accumulator and writes
row shard c of dW = scale * sum_r dW_r to dw_shards[c].  Compared with the fp64
oracle (normwise relative error <= 1e-2; exact for integer-valued operands).
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


def to_dev(bits):
    return workloads.bits_to_torch_bf16(bits).to(DEV)


def rel_err(y, ref):
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def run(K, T, F, D, dt, ints=False, scale=None):
    dys, xs = workloads.wgrad_operands(T, F, D, K, ints=ints)
    shards = col.wgrad_reduce_scatter([to_dev(a) for a in dys], [to_dev(a) for a in xs],
                                      scale, dt)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    got = torch.cat(shards, dim=0).double().cpu().numpy()
    return dys, xs, got


@pytest.mark.parametrize("K,T,F,D,dt", [
    (8, 64, 1024, 256, torch.bfloat16),    # shards of 128 rows: TMA-store epilogue
    (4, 100, 256, 192, torch.float32),     # ragged tokens, D a multiple of 64 only
    (2, 256, 128, 512, torch.bfloat16),    # several token blocks per rank
    (1, 130, 128, 64, torch.float32),      # K = 1: a plain dy^T x
    (16, 32, 256, 128, torch.bfloat16),    # 16-row shards: per-thread epilogue
    (8, 1, 512, 64, torch.float32),        # one token per rank
    (3, 70, 192, 320, torch.bfloat16),     # three ranks, ragged everything
])
def test_shapes_against_fp64(K, T, F, D, dt):
    dys, xs, got = run(K, T, F, D, dt)
    ref = oracle.wgrad_psum_f64(dys, xs, 1.0 / K)
    assert got.shape == ref.shape
    assert rel_err(got, ref) <= TOL


@pytest.mark.parametrize("K,T,F,D", [(8, 64, 128, 128), (4, 128, 256, 64), (2, 256, 64, 192)])
def test_integer_operands_are_exact(K, T, F, D):
    # |values| <= 4 and at most 512 products per output: every partial sum
    # is an integer below 2^24, so fp32 accumulation is exact in any order
    dys, xs, got = run(K, T, F, D, torch.float32, ints=True, scale=1.0)
    assert np.array_equal(got, oracle.wgrad_psum_f64(dys, xs))


def test_zero_tokens_give_zero_gradient():
    K, F, D = 4, 128, 64
    outs = [torch.full((F // K, D), 7.0, device=DEV) for _ in range(K)]
    dyp = [torch.empty(16, F, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    xp = [torch.empty(16, D, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    B.dp_wgrad_reduce_scatter(dyp, xp, K, 0, F, D, outs, B.DP_FP32, 0.25)
    torch.cuda.synchronize()
    assert all(bool((o == 0).all()) for o in outs)


def test_repeated_calls_are_deterministic():
    dys, xs = workloads.wgrad_operands(200, 256, 128, 4)
    d, x = [to_dev(a) for a in dys], [to_dev(a) for a in xs]
    a = col.wgrad_reduce_scatter(d, x, 0.25, torch.float32)
    b = col.wgrad_reduce_scatter(d, x, 0.25, torch.float32)
    assert all(torch.equal(p, q) for p, q in zip(a, b))


def test_rejects_unsupported_shapes():
    d = [torch.zeros(16, 128, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    x = [torch.zeros(16, 64, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    o = [torch.zeros(16, 64, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    st = B.dp_wgrad_reduce_scatter(d, x, 8, 16, 96, 64, o, B.DP_BF16, 1.0, check=False)
    assert st == B.DP_ERR_UNSUPPORTED  # F % 64 != 0
    st = B.dp_wgrad_reduce_scatter(d[:5], x[:5], 5, 16, 128, 64, o[:5], B.DP_BF16, 1.0,
                                   check=False)
    assert st == B.DP_ERR_INVALID_ARG  # F % K


def test_full_size_sampled():
    """8 ranks x 1024 tokens, dy [1024, 4096] and x [1024, 4096] -> dW [4096,
    4096] in eight [512, 4096] shards (the benchmark's launch configuration);
    sampled outputs against the fp64 oracle."""
    K, T, F, D = 8, 1024, 4096, 4096
    dys, xs = workloads.wgrad_operands(T, F, D, K)
    shards = col.wgrad_reduce_scatter([to_dev(a) for a in dys], [to_dev(a) for a in xs],
                                      1.0 / K, torch.bfloat16)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    rng = np.random.default_rng(7)
    fs = np.concatenate([rng.integers(0, F, 1500), [0, F - 1, 511, 512]])
    ds = np.concatenate([rng.integers(0, D, 1500), [0, D - 1, 255, 256]])
    ref = oracle.wgrad_psum_f64_sampled(dys, xs, fs, ds, 1.0 / K)
    rows = F // K
    got = np.array([float(shards[f // rows][f % rows, d]) for f, d in zip(fs, ds)])
    assert rel_err(got, ref) <= TOL
    assert all(bool(torch.isfinite(s).all()) for s in shards)


# ---- chained split of the last round through a workspace --------------------
#
# With a workspace, the tiles of a last, less-than-half-full round of the
# persistent grid are cut into token-block segments on different CTAs, each
# continuing the previous one's fp32 accumulator.  Every element sees the same
# MMAs in the same order, so the output must be bitwise the one without the
# split.  CTA limits make small problems take the split with 2, 3 and 4
# segments (the segment that starts a CTA's list, one in the middle, one at
# its end).

def _limits(gemm):
    B.dp_set_cta_limits(gemm, 0)


@pytest.fixture
def restore_limits():
    g, s = B.dp_get_cta_limits()
    yield
    B.dp_set_cta_limits(g, s)


def _run_ws(dys, xs, K, T, F, D, dt, ws):
    out = [torch.full((F // K, D), float("nan"), dtype=dt, device=DEV) for _ in range(K)]
    B.dp_wgrad_reduce_scatter(dys, xs, K, T, F, D, out, col._DT[dt], 1.0 / K, workspace=ws)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    return out


def _bits(ts):
    return [t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32) for t in ts]


@pytest.mark.parametrize("limit,K,T,F,D,dt", [
    (10, 4, 256, 512, 512, torch.bfloat16),   # 32 tiles on 10 CTAs: 2 tail tiles, 2 segments
    (10, 4, 512, 512, 512, torch.float32),    # 4 segments (slots 0..3)
    (15, 4, 512, 512, 512, torch.bfloat16),   # 3 segments (slots 0, 1, 2)
    (4, 4, 200, 256, 320, torch.float32),     # ragged token blocks, 64-wide tiles
    (6, 2, 512, 256, 256, torch.bfloat16),    # 8 tiles on 6 CTAs
    (6, 1, 1024, 256, 256, torch.float32),    # one rank: a plain dy^T x, split
])
def test_split_is_bitwise_the_unsplit_result(restore_limits, limit, K, T, F, D, dt):
    dys_h, xs_h = workloads.wgrad_operands(T, F, D, K)
    dys, xs = [to_dev(a) for a in dys_h], [to_dev(a) for a in xs_h]
    _limits(limit)
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    assert need > 0  # the shape splits under this limit
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    plain = _run_ws(dys, xs, K, T, F, D, dt, None)
    split = _run_ws(dys, xs, K, T, F, D, dt, ws)
    again = _run_ws(dys, xs, K, T, F, D, dt, ws)  # flags were cleared by the first
    for a, b, c in zip(_bits(plain), _bits(split), _bits(again)):
        assert torch.equal(a, b) and torch.equal(a, c)
    _limits(0)
    nolimit = _run_ws(dys, xs, K, T, F, D, dt, None)
    for a, b in zip(_bits(plain), _bits(nolimit)):
        assert torch.equal(a, b)
    ref = oracle.wgrad_psum_f64(dys_h, xs_h, 1.0 / K)
    got = torch.cat(split, dim=0).double().cpu().numpy()
    assert rel_err(got, ref) <= TOL


def test_split_with_integer_operands_is_exact(restore_limits):
    K, T, F, D = 2, 512, 256, 256
    dys_h, xs_h = workloads.wgrad_operands(T, F, D, K, ints=True)
    _limits(6)
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = [torch.empty(F // K, D, device=DEV) for _ in range(K)]
    B.dp_wgrad_reduce_scatter([to_dev(a) for a in dys_h], [to_dev(a) for a in xs_h], K, T, F, D,
                              out, B.DP_FP32, 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    got = torch.cat(out, dim=0).double().cpu().numpy()
    assert np.array_equal(got, oracle.wgrad_psum_f64(dys_h, xs_h))


def test_too_small_workspace_runs_unsplit(restore_limits):
    K, T, F, D = 4, 256, 512, 512
    dys_h, xs_h = workloads.wgrad_operands(T, F, D, K)
    dys, xs = [to_dev(a) for a in dys_h], [to_dev(a) for a in xs_h]
    _limits(10)
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    a = _run_ws(dys, xs, K, T, F, D, torch.bfloat16, None)
    b = _run_ws(dys, xs, K, T, F, D, torch.bfloat16, small)
    assert all(torch.equal(p, q) for p, q in zip(_bits(a), _bits(b)))


def test_no_split_needs_no_workspace(restore_limits):
    _limits(0)
    assert B.dp_wgrad_workspace_size(4, 128, 256, 128) == 0  # fewer tiles than SMs
    assert B.dp_wgrad_workspace_size(8, 0, 4096, 4096) == 0  # no tokens
    _limits(8)
    assert B.dp_wgrad_workspace_size(4, 512, 512, 512) == 0  # 32 tiles fill 8 CTAs 4 times


def test_split_in_a_cuda_graph_follows_new_inputs(restore_limits):
    # replays reuse the launch's flag value; each flag is cleared once read,
    # so a replay never reads a hand-off of the previous one
    K, T, F, D = 4, 512, 512, 512
    _limits(10)
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    sets = [workloads.wgrad_operands(T, F, D, K, std=s) for s in (0.02, 0.05, 0.01)]
    dys = [torch.empty(T, F, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    xs = [torch.empty(T, D, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    out = [torch.empty(F // K, D, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside capture (tensor maps encoded)
        B.dp_wgrad_reduce_scatter(dys, xs, K, T, F, D, out, B.DP_BF16, 0.25, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.dp_wgrad_reduce_scatter(dys, xs, K, T, F, D, out, B.DP_BF16, 0.25, workspace=ws)
    for dh, xh in sets:
        for r in range(K):
            dys[r].copy_(to_dev(dh[r]))
            xs[r].copy_(to_dev(xh[r]))
        g.replay()
        torch.cuda.synchronize()
        assert B.dp_get_device_error() == B.DP_OK
        want = _run_ws(dys, xs, K, T, F, D, torch.bfloat16, None)
        assert all(torch.equal(p, q) for p, q in zip(_bits(out), _bits(want)))


def test_full_size_split_is_bitwise_the_unsplit_result(restore_limits):
    """The benchmark's shape: 512 tiles on 152 SMs leave 56 for a fourth
    round, which runs as two chained halves."""
    _limits(0)
    K, T, F, D = 8, 1024, 4096, 4096
    dys_h, xs_h = workloads.wgrad_operands(T, F, D, K)
    dys, xs = [to_dev(a) for a in dys_h], [to_dev(a) for a in xs_h]
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (F // 128) * (D // 256)
    if 0 < tiles % n_sm <= n_sm // 2:
        assert need > 0
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)
    a = _run_ws(dys, xs, K, T, F, D, torch.bfloat16, None)
    b = _run_ws(dys, xs, K, T, F, D, torch.bfloat16, ws)
    assert all(torch.equal(p, q) for p, q in zip(_bits(a), _bits(b)))
