"""GPU parity of the DDP bucket all-reduce (in place, no flattening) and of
the Reducer driving it, bit for bit against the oracle's ring all-reduce of
the flattened bucket."""
import random

import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col
from tests.test_reducer_cpu import expected_buckets

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def rand_tensors(K, sizes, dt, seed):
    rng = np.random.default_rng(seed)
    host = []
    for r in range(K):
        row = []
        for n in sizes:
            a = rng.uniform(-1, 1, n).astype(np.float32)
            row.append(workloads.to_bf16_bits(a) if dt == "bf16" else a)
        host.append(row)
    return host


def to_dev(a, offset=0):
    t = workloads.bits_to_torch_bf16(a) if a.dtype == np.uint16 else torch.from_numpy(a)
    if offset == 0:
        return t.to(DEV)
    raw = torch.empty(a.size + offset, dtype=t.dtype, device=DEV)
    raw[offset:].copy_(t)
    return raw[offset:]


def bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


def as_bits(a):
    return a.view(np.int16) if a.dtype == np.uint16 else a.view(np.int32)


@pytest.mark.parametrize("K", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("offset", [0, 1])
def test_bucket_allreduce_matches_oracle(K, dt, offset):
    sizes = [1, 7, 8, 1000, 4099, 16, 33, 8 * 1237, 5]
    host = rand_tensors(K, sizes, dt, 7 * K + offset)
    dev = [[to_dev(a, offset) for a in row] for row in host]
    col.bucket_allreduce_(dev, 1.0 / K)
    torch.cuda.synchronize()
    ref = oracle.bucket_all_reduce(host, 1.0 / K)
    for r in range(K):
        for t in range(len(sizes)):
            assert np.array_equal(bits(dev[r][t]), as_bits(ref[r][t])), (r, t)


def test_bucket_with_many_tensors_spans_launches():
    K, n = 4, 300  # more tensors than one launch's parameter table holds
    rng = random.Random(3)
    sizes = [rng.randint(1, 3000) for _ in range(n)]
    host = rand_tensors(K, sizes, "f32", 11)
    dev = [[to_dev(a) for a in row] for row in host]
    col.bucket_allreduce_(dev, 0.25)
    ref = oracle.bucket_all_reduce(host, 0.25)
    for r in range(K):
        for t in range(n):
            assert np.array_equal(bits(dev[r][t]), as_bits(ref[r][t]))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_reducer_end_to_end_shuffled_ready_order(dt):
    K = 4
    rng = random.Random(5)
    numels = [rng.choice([64, 768, 3000, 4096, 65536, 100003]) for _ in range(40)]
    esize = 4 if dt == "f32" else 2
    cap = 256 * 1024
    host = rand_tensors(K, numels, dt, 9)
    dev = [[to_dev(a) for a in row] for row in host]
    red = col.Reducer(numels, B.DP_FP32 if dt == "f32" else B.DP_BF16, K,
                      bucket_cap_bytes=cap, scale=1.0 / K)
    order = list(range(len(numels)))[::-1]
    rng.shuffle(order)  # backward hooks fire in no particular order
    for p in order:
        red.mark_ready(p, [dev[r][p] for r in range(K)])
    assert red.finish() == (B.DP_OK, -1)
    torch.cuda.synchronize()
    for members in expected_buckets(numels, esize, cap):
        ref = oracle.bucket_all_reduce([[host[r][p] for p in members] for r in range(K)], 1.0 / K)
        for r in range(K):
            for i, p in enumerate(members):
                assert np.array_equal(bits(dev[r][p]), as_bits(ref[r][i])), (p, r)


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("K,sizes", [(2, [3, 21]), (3, [5, 40, 17, 64]), (4, [1, 2, 3, 4, 8000, 9])])
def test_chunk_boundary_inside_a_vector(variant, K, sizes):
    """Bucket offsets that are not multiples of 8 put ring-chunk boundaries
    inside 16-byte vectors: those elements fold in their own chunk's order."""
    host = rand_tensors(K, sizes, "f32", 41 + K)
    dev = [[to_dev(a) for a in row] for row in host]
    B.dp_set_collective_variant(variant)
    try:
        col.bucket_allreduce_(dev, 1.0 / K)
        torch.cuda.synchronize()
    finally:
        B.dp_set_collective_variant(0)
    ref = oracle.bucket_all_reduce(host, 1.0 / K)
    for r in range(K):
        for t in range(len(sizes)):
            assert np.array_equal(bits(dev[r][t]), as_bits(ref[r][t])), (r, t)


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("K", [3, 8])
def test_empty_tensors_take_no_part(variant, K):
    # zero-size tensors (whose data pointer may be NULL) anywhere in a bucket
    sizes = [0, 5, 0, 4099, 0, 8, 16 * 1000 + 3, 0]
    host = rand_tensors(K, sizes, "f32", 61 + K)
    dev = [[to_dev(a) for a in row] for row in host]
    B.dp_set_collective_variant(variant)
    try:
        col.bucket_allreduce_(dev, 1.0 / K)
    finally:
        B.dp_set_collective_variant(0)
    torch.cuda.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    ref = oracle.bucket_all_reduce(host, 1.0 / K)
    for r in range(K):
        for t in range(len(sizes)):
            assert np.array_equal(bits(dev[r][t]), as_bits(ref[r][t])), (r, t)


def test_reducer_with_empty_parameters():
    K = 4
    numels = [100, 0, 64, 0, 3000, 0]
    host = rand_tensors(K, numels, "f32", 71)
    dev = [[to_dev(a) for a in row] for row in host]
    red = col.Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=1024, scale=0.25)
    for p in reversed(range(len(numels))):
        red.mark_ready(p, [dev[r][p].data_ptr() for r in range(K)])
    st, first_pending = red.finish()
    assert st == B.DP_OK and first_pending == -1
    torch.cuda.synchronize()
    for members in expected_buckets(numels, 4, 1024):
        ref = oracle.bucket_all_reduce([[host[r][p] for p in members] for r in range(K)], 0.25)
        for r in range(K):
            for i, p in enumerate(members):
                assert np.array_equal(bits(dev[r][p]), as_bits(ref[r][i]))



@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_reducer_overlap_reduces_beside_the_backward(dt):
    """DDP's asynchronous all-reduce: in overlap mode each bucket is reduced
    on the reducer's own stream while the caller's stream goes on with the
    "backward" -- here, writing the next parameters' gradients and a GEMM per
    parameter to keep it busy.  The buckets read gradients written on the
    caller's stream just before they completed, so the results also check
    the events between the streams: bit for bit against the oracle, and
    equal to the same iteration without overlap."""
    K = 4
    rng = random.Random(6)
    numels = [rng.choice([64, 768, 3000, 4096, 65536, 100003]) for _ in range(30)]
    esize = 4 if dt == "f32" else 2
    cap = 256 * 1024
    host = rand_tensors(K, numels, dt, 12)
    src = [[to_dev(a) for a in row] for row in host]
    dev = [[torch.full_like(t, float("nan")) for t in row] for row in src]
    red = col.Reducer(numels, B.DP_FP32 if dt == "f32" else B.DP_BF16, K,
                      bucket_cap_bytes=cap, scale=1.0 / K)
    red.set_overlap(True)
    x, ws = workloads.gemm_operands(1024, 1024, 8, 128)
    xd = workloads.bits_to_torch_bf16(x).to(DEV)
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for it in range(2):  # two iterations through the same reducer
            for p in reversed(range(len(numels))):  # backward order
                col.allgather_matmul(xd, wd, stream=s)
                for r in range(K):
                    dev[r][p].copy_(src[r][p])
                red.mark_ready(p, [dev[r][p] for r in range(K)], stream=s)
            red.wait(stream=s)
            assert red.finish() == (B.DP_OK, -1)
            if it == 0:
                first = [[bits(t) for t in row] for row in dev]
    s.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    for members in expected_buckets(numels, esize, cap):
        ref = oracle.bucket_all_reduce([[host[r][p] for p in members] for r in range(K)], 1.0 / K)
        for r in range(K):
            for i, p in enumerate(members):
                assert np.array_equal(bits(dev[r][p]), as_bits(ref[r][i])), (p, r)
                assert np.array_equal(first[r][p], as_bits(ref[r][i])), (p, r)
    red.set_overlap(False)


def test_reducer_overlap_in_a_cuda_graph():
    """One overlapped Reducer iteration captured in a CUDA graph: the bucket
    launches on the Reducer's stream fork from and join back to the
    capturing stream through its events; replays give the oracle's bits."""
    K = 4
    rng = random.Random(8)
    numels = [rng.choice([64, 768, 3000, 4096, 65536]) for _ in range(24)]
    cap = 128 * 1024
    host = rand_tensors(K, numels, "f32", 13)
    src = [[to_dev(a) for a in row] for row in host]
    dev = [[torch.empty_like(t) for t in row] for row in src]
    red = col.Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=cap, scale=1.0 / K)
    red.set_overlap(True)
    s = torch.cuda.Stream()

    def iteration():
        for p in reversed(range(len(numels))):
            for r in range(K):
                dev[r][p].copy_(src[r][p])
            red.mark_ready(p, [dev[r][p] for r in range(K)], stream=s)
        red.wait(stream=s)
        assert red.finish() == (B.DP_OK, -1)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):  # once eagerly (kernel attributes set up outside capture)
        iteration()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        iteration()
    for _ in range(2):
        for row in dev:
            for t in row:
                t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for members in expected_buckets(numels, 4, cap):
            ref = oracle.bucket_all_reduce([[host[r][p] for p in members] for r in range(K)],
                                           1.0 / K)
            for r in range(K):
                for i, p in enumerate(members):
                    assert np.array_equal(bits(dev[r][p]), as_bits(ref[r][i])), (p, r)
    assert B.dp_get_device_error() == B.DP_OK
    red.set_overlap(False)


@pytest.mark.parametrize("K,numels,cap", [
    (2, [5000, 3, 77], 1 << 30),                  # one bucket: the second stream stays idle
    (3, [4096] * 5, 4096 * 4),                    # five buckets: the streams end unevenly
    (8, [1, 8, 100003, 16, 4099, 8 * 1237], 1024),  # a bucket per tensor, tiny and ragged
])
def test_reducer_overlap_bucket_counts(K, numels, cap):
    """Overlap mode alternates buckets over the Reducer's two streams; the
    join covers both whatever the bucket count, and a bucket that starts
    while the previous one (on the other stream) still runs gives the
    oracle's bits."""
    host = rand_tensors(K, numels, "f32", 31 + K)
    dev = [[to_dev(a) for a in row] for row in host]
    red = col.Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=cap, scale=1.0 / K)
    red.set_overlap(True)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for p in reversed(range(len(numels))):
            red.mark_ready(p, [dev[r][p] for r in range(K)], stream=s)
        red.wait(stream=s)
        assert red.finish() == (B.DP_OK, -1)
        # reads on the caller's stream after the join see every bucket
        got = [[t.clone() for t in row] for row in dev]
    s.synchronize()
    assert B.dp_get_device_error() == B.DP_OK
    for members in expected_buckets(numels, 4, cap):
        ref = oracle.bucket_all_reduce([[host[r][p] for p in members] for r in range(K)], 1.0 / K)
        for r in range(K):
            for i, p in enumerate(members):
                assert np.array_equal(bits(got[r][p]), as_bits(ref[r][i])), (p, r)
    red.set_overlap(False)
