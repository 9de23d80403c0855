"""The bulk-copy (shared-memory staged, cp.async.bulk) variant of the
all-reduce and all-gather: bit-identical to the oracle and to the register
variant, including ragged chunk tails, partial tiles and K=16 (the largest
shared-memory footprint)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture
def bulk():
    B.dp_set_collective_variant(2)
    try:
        yield
    finally:
        B.dp_set_collective_variant(0)


def host_bufs(K, N, dt, seed):
    rng = np.random.default_rng(seed)
    f = [rng.uniform(-1, 1, N).astype(np.float32) for _ in range(K)]
    return [workloads.to_bf16_bits(a) for a in f] if dt == "bf16" else f


def to_dev(a):
    t = workloads.bits_to_torch_bf16(a) if a.dtype == np.uint16 else torch.from_numpy(a)
    return t.to(DEV)


def bits(t):
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


def as_bits(a):
    return a.view(np.int16) if a.dtype == np.uint16 else a.view(np.int32)


@pytest.mark.parametrize("K", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N", [8 * 5000, 8 * 8 * 1024 * 3 + 8 * 40, 8 * 64 * 1000 - 13])
def test_bulk_allreduce_matches_oracle(bulk, K, dt, N):
    if N % 8 and K == 1:
        pytest.skip("covered by the K>1 ragged cases")
    host = host_bufs(K, N, dt, 3 * K + N)
    bufs = [to_dev(h) for h in host]
    col.all_reduce_(bufs, 1.0 / K)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    ref = oracle.all_reduce(host, 1.0 / K)
    for r in range(K):
        assert np.array_equal(bits(bufs[r]), as_bits(ref[r])), r


@pytest.mark.parametrize("K", [2, 8, 16])
@pytest.mark.parametrize("dt,C", [("f32", 4 * 10000), ("bf16", 8 * 3333), ("f32", 4 * 4096 * 5)])
def test_bulk_all_gather_matches_oracle(bulk, K, dt, C):
    host = host_bufs(K, C, dt, K + C)
    shards = [to_dev(h) for h in host]
    out = col.all_gather(shards)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    ref = oracle.all_gather(host)
    for r in range(K):
        assert np.array_equal(bits(out[r]), as_bits(ref[r]))


@pytest.mark.parametrize("K", [1, 3, 5, 16])
@pytest.mark.parametrize("cap", [0, 8, 40])
@pytest.mark.parametrize("dt,C", [("f32", 16384 * 3 + 12), ("bf16", 16)])
def test_bulk_all_gather_schedules_match_oracle(bulk, K, cap, dt, C):
    """Both schedules of the bulk-copy all-gather: one destination rank per
    CTA (the whole GPU) and one source shard per CTA (a CTA cap, as a
    collective beside a GEMM gets); shards of 3 tiles and 48 bytes, and of
    32 bytes, for odd rank counts."""
    host = host_bufs(K, C, dt, 7 * K + C)
    shards = [to_dev(h) for h in host]
    saved = B.dp_get_cta_limits()
    try:
        B.dp_set_cta_limits(saved[0], cap)
        out = col.all_gather(shards)
        torch.cuda.synchronize()
    finally:
        B.dp_set_cta_limits(*saved)
    assert B.dp_get_device_error() == B.DP_OK
    ref = oracle.all_gather(host)
    for r in range(K):
        assert np.array_equal(bits(out[r]), as_bits(ref[r]))


def test_variants_agree_at_full_size():
    K, N = 8, 64 * 1024 * 1024
    base = workloads.sweep_bufs_device(K, N, DEV)
    a = [t.clone() for t in base]
    b = [t.clone() for t in base]
    B.dp_set_collective_variant(1)
    try:
        col.all_reduce_(a, 1.0 / K)
        g1 = col.all_gather([t[: N // K] for t in base])
        B.dp_set_collective_variant(2)
        col.all_reduce_(b, 1.0 / K)
        g2 = col.all_gather([t[: N // K] for t in base])
    finally:
        B.dp_set_collective_variant(0)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    for r in range(K):
        assert torch.equal(a[r].view(torch.int32), b[r].view(torch.int32))
        assert torch.equal(g1[r].view(torch.int32), g2[r].view(torch.int32))


def test_variant_switch_rejects_unknown_values():
    assert B.dp_set_collective_variant(3, check=False) == B.DP_ERR_INVALID_ARG
    assert B.dp_get_collective_variant() == 0


@pytest.mark.parametrize("K", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("C", [8 * 3001, 2048 * 5, 8])
@pytest.mark.parametrize("outs", [("f32", "bf16"), ("f32",), ("bf16",)])
def test_bulk_reduce_scatter_matches_oracle(bulk, K, dt, C, outs):
    N = K * C
    host = host_bufs(K, N, dt, 11 * K + C)
    bufs = [to_dev(h) for h in host]
    o32, o16 = col.reduce_scatter(bufs, 1.0 / K, outs)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    r32, r16 = oracle.reduce_scatter(host, 1.0 / K)
    for c in range(K):
        if o32 is not None:
            assert np.array_equal(bits(o32[c]), as_bits(r32[c]))
        if o16 is not None:
            assert np.array_equal(bits(o16[c]), as_bits(r16[c]))


def test_bulk_reduce_scatter_full_size_equals_register_variant():
    K, N = 8, 64 * 1024 * 1024
    bufs = workloads.fsdp_grads_device(K, N, DEV)
    B.dp_set_collective_variant(1)
    try:
        a32, a16 = col.reduce_scatter(bufs, 1.0 / K)
        B.dp_set_collective_variant(2)
        b32, b16 = col.reduce_scatter(bufs, 1.0 / K)
    finally:
        B.dp_set_collective_variant(0)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    for c in range(K):
        assert torch.equal(a32[c].view(torch.int32), b32[c].view(torch.int32))
        assert torch.equal(a16[c].view(torch.int16), b16[c].view(torch.int16))
