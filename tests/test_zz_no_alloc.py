"""GPU test of dp_wgrad_reduce_scatter_noalloc, the weight-gradient
reduce-scatter for callers that cannot allocate device memory (a framework
pool that owns the GPU, a step that cannot take cudaMalloc's device-wide
synchronisation, a memory budget fixed at start-up).  It takes its scratch
from a device array built into the library instead of a caller's workspace.

Through the C ABI, two calls in a row on the benchmark's shape (whose last
round is split through that scratch) and on a small shape split into four
segments under a CTA limit, each checked against the existing entry point
with a caller-allocated workspace: within the fp64 tolerance of the other
weight-gradient tests against the oracle, and bit for bit against each
other.  A shape that would need more scratch than the built-in array is
rejected before anything is launched.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TOL = 1e-2


def to_dev(bits):
    return workloads.bits_to_torch_bf16(bits).to(DEV)


@pytest.fixture
def cta_limit():
    saved = B.dp_get_cta_limits()

    def set_gemm(n):
        B.dp_set_cta_limits(n, 0)

    yield set_gemm
    B.dp_set_cta_limits(*saved)


def _outs(K, F, D):
    return [torch.full((F // K, D), float("nan"), dtype=torch.bfloat16, device=DEV)
            for _ in range(K)]


def _bits(ts):
    return [t.view(torch.int16) for t in ts]


def _check(K, T, F, D, sampled):
    dys_h, xs_h = workloads.wgrad_operands(T, F, D, K)
    dys, xs = [to_dev(a) for a in dys_h], [to_dev(a) for a in xs_h]
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    assert 0 < need <= B.DP_WGRAD_NOALLOC_MAX_BYTES  # the shape uses the scratch
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    want = _outs(K, F, D)
    B.dp_wgrad_reduce_scatter(dys, xs, K, T, F, D, want, B.DP_BF16, 1.0 / K, workspace=ws)
    for _ in range(2):
        got = _outs(K, F, D)
        assert B.dp_wgrad_reduce_scatter_noalloc(dys, xs, K, T, F, D, got, B.DP_BF16,
                                                 1.0 / K) == B.DP_OK
        torch.cuda.synchronize()
        assert B.dp_get_device_error() == B.DP_OK
        g = torch.cat(got).double()
        w = torch.cat(want).double()
        assert float(torch.linalg.norm(g - w) / torch.linalg.norm(w)) <= TOL
        assert all(torch.equal(a, b) for a, b in zip(_bits(got), _bits(want)))
    rows = F // K
    if sampled:
        rng = np.random.default_rng(3)
        fs, ds = rng.integers(0, F, 600), rng.integers(0, D, 600)
        ref = oracle.wgrad_psum_f64_sampled(dys_h, xs_h, fs, ds, 1.0 / K)
        val = np.array([float(got[f // rows][f % rows, d]) for f, d in zip(fs, ds)])
    else:
        ref = oracle.wgrad_psum_f64(dys_h, xs_h, 1.0 / K)
        val = torch.cat(got).double().cpu().numpy()
    assert np.linalg.norm(val - ref) / np.linalg.norm(ref) <= TOL


def test_noalloc_matches_the_workspace_call_at_bench_size(cta_limit):
    cta_limit(0)
    K, T, F, D = 8, 1024, 4096, 4096
    if B.dp_wgrad_workspace_size(K, T, F, D) == 0:
        pytest.skip("this GPU's SM count leaves no part-full last round for this shape")
    _check(K, T, F, D, sampled=True)


def test_noalloc_matches_the_workspace_call_four_segments(cta_limit):
    cta_limit(10)  # 32 tiles on 10 CTAs: two tail tiles in four segments
    _check(4, 512, 512, 512, sampled=False)


def test_noalloc_fp32_output_matches_the_workspace_call(cta_limit):
    cta_limit(10)
    K, T, F, D = 4, 512, 512, 512
    dys_h, xs_h = workloads.wgrad_operands(T, F, D, K)
    dys, xs = [to_dev(a) for a in dys_h], [to_dev(a) for a in xs_h]
    need = B.dp_wgrad_workspace_size(K, T, F, D)
    assert 0 < need <= B.DP_WGRAD_NOALLOC_MAX_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    want = [torch.empty(F // K, D, device=DEV) for _ in range(K)]
    B.dp_wgrad_reduce_scatter(dys, xs, K, T, F, D, want, B.DP_FP32, 0.25, workspace=ws)
    for _ in range(2):
        got = [torch.full((F // K, D), float("nan"), device=DEV) for _ in range(K)]
        assert B.dp_wgrad_reduce_scatter_noalloc(dys, xs, K, T, F, D, got, B.DP_FP32,
                                                 0.25) == B.DP_OK
        torch.cuda.synchronize()
        assert B.dp_get_device_error() == B.DP_OK
        assert all(torch.equal(a.view(torch.int32), b.view(torch.int32))
                   for a, b in zip(got, want))


def test_noalloc_rejects_more_than_its_scratch(cta_limit):
    # 512 tiles on 148 CTAs leave 68 in halves: 68 x 128 KiB > 8 MiB
    K, T, F, D = 8, 1024, 4096, 4096
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    if n_sm < 148:
        pytest.skip("needs 148 SMs")
    cta_limit(148)
    assert B.dp_wgrad_workspace_size(K, T, F, D) > B.DP_WGRAD_NOALLOC_MAX_BYTES
    d = [torch.zeros(T, F, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    x = [torch.zeros(T, D, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    o = [torch.full((F // K, D), 3.0, dtype=torch.bfloat16, device=DEV) for _ in range(K)]
    st = B.dp_wgrad_reduce_scatter_noalloc(d, x, K, T, F, D, o, B.DP_BF16, 1.0, check=False)
    assert st == B.DP_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert all(bool((t == 3.0).all()) for t in o)  # nothing was launched
