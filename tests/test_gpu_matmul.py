"""GPU parity of the fused all-gather + GEMM (tcgen05) against the fp64 oracle.

The bar: normwise relative error ||y - y_ref||_F / ||y_ref||_F <= 1e-2; with
integer-valued operands (every fp32 partial sum exact) the fp32 output must be
exact.  Shapes cover the FSDP fixture, several tiles with ragged M and D,
shard widths that need one or several TMA boxes per tile, and the full
x[8192,4096] . w[4096,4096]^T workload on sampled outputs.
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


def run(M, D, K, F_shard, y_dtype=torch.bfloat16, ints=False):
    if ints:
        x, ws = workloads.gemm_int_operands(M, D, K, F_shard)
    else:
        x, ws = workloads.gemm_operands(M, D, K, F_shard)
    y = col.allgather_matmul(to_dev(x), [to_dev(w) for w in ws], y_dtype)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    return x, ws, y.double().cpu().numpy()


def test_fsdp_fixture_128x512_against_fp64():
    x, ws, y = run(128, 512, 8, 64, torch.float32)
    ref = oracle.allgather_matmul_f64(x, ws)
    assert rel_err(y, ref) <= TOL
    # fp32 accumulation of 512 products: far tighter than the bar
    assert rel_err(y, ref) <= 1e-5


def test_fsdp_fixture_bf16_output():
    x, ws, y = run(128, 512, 8, 64, torch.bfloat16)
    ref = oracle.allgather_matmul_f64(x, ws)
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("M,D,K,F_shard", [(256, 512, 8, 64), (384, 256, 4, 128),
                                           (128, 512, 2, 512), (256, 128, 16, 16)])
def test_integer_operands_are_exact(M, D, K, F_shard):
    x, ws, y = run(M, D, K, F_shard, torch.float32, ints=True)
    ref = oracle.allgather_matmul_f64(x, ws)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("M,D,K,F_shard,ydt", [
    (200, 512, 8, 64, torch.bfloat16),    # ragged M
    (256, 72, 8, 64, torch.float32),      # ragged D (k-block tail)
    (130, 136, 3, 48, torch.float32),     # shard width not a power of two
    (512, 1024, 4, 512, torch.bfloat16),  # several k-blocks, one shard per tile
    (1024, 256, 1, 256, torch.float32),   # K = 1: a plain GEMM
    (64, 256, 16, 32, torch.bfloat16),    # M below one tile, many narrow shards
    (1280, 640, 8, 320, torch.float32),   # F_shard > 256, not a multiple of 256
])
def test_shapes_against_fp64(M, D, K, F_shard, ydt):
    x, ws, y = run(M, D, K, F_shard, ydt)
    ref = oracle.allgather_matmul_f64(x, ws)
    assert y.shape == ref.shape
    assert rel_err(y, ref) <= TOL


def test_repeated_calls_are_deterministic():
    x, ws = workloads.gemm_operands(512, 512, 8, 128)
    xt, wt = to_dev(x), [to_dev(w) for w in ws]
    a = col.allgather_matmul(xt, wt, torch.float32)
    b = col.allgather_matmul(xt, wt, torch.float32)
    assert torch.equal(a, b)


def test_full_size_sampled():
    """x[8192,4096], 8 shards w_k[512,4096] -> y[8192,4096]: sampled outputs
    against the fp64 oracle, in the benchmark's launch configuration."""
    M, D, K, F_shard = 8192, 4096, 8, 512
    x, ws = workloads.gemm_operands(M, D, K, F_shard)
    y = col.allgather_matmul(to_dev(x), [to_dev(w) for w in ws], torch.bfloat16)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    rng = np.random.default_rng(1)
    ms = np.concatenate([rng.integers(0, M, 1500), [0, M - 1, 127, 128]])
    fs = np.concatenate([rng.integers(0, K * F_shard, 1500), [0, K * F_shard - 1, 511, 512]])
    ref = oracle.allgather_matmul_f64_sampled(x, ws, ms, fs)
    got = y[torch.from_numpy(ms).to(DEV), torch.from_numpy(fs).to(DEV)].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL
    # every output is finite and the product is not trivially zero
    assert torch.isfinite(y).all()
    assert float(y.float().abs().mean()) > 0
