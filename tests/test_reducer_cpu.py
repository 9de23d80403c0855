"""Host logic of the DDP gradient Reducer, without a GPU (dry-run mode records
bucket launches instead of launching kernels).

The rules come from "CMU 11-868 L14-L15 ...", sections "When to sync:
gradient bucketing" and "What the paper adds beyond the slides": buckets are
filled in reverse parameter order up to the size cap, fixed at construction;
a bucket is all-reduced once all its gradients are ready; buckets go out
strictly in order; an unused parameter leaves its bucket incomplete (DDP
would hang; the Reducer reports it).
"""
import random

import pytest

from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import build as cuda_build
from ring_allreduce_gradient_gb300.collectives import Reducer

MB = 1024 * 1024


@pytest.fixture(scope="module", autouse=True)
def lib():
    cuda_build.build()
    B.load()


def expected_buckets(numels, esize, cap):
    """The size rule restated: walk parameters last to first, close a bucket
    once its bytes reach the cap."""
    buckets, cur, size = [], [], 0
    for p in reversed(range(len(numels))):
        cur.append(p)
        size += numels[p] * esize
        if size >= cap:
            buckets.append(cur)
            cur, size = [], 0
    if cur:
        buckets.append(cur)
    return buckets


@pytest.mark.parametrize("cap_mb", [1, 25, 100])
def test_bucket_assignment_follows_the_size_rule(cap_mb):
    rng = random.Random(cap_mb)
    numels = [rng.choice([768, 3072, 768 * 768, 768 * 3072, 50257 * 768]) for _ in range(60)]
    r = Reducer(numels, B.DP_FP32, K=8, bucket_cap_bytes=cap_mb * MB)
    exp = expected_buckets(numels, 4, cap_mb * MB)
    assert r.num_buckets == len(exp)
    for b, members in enumerate(exp):
        n, ne = r.bucket_info(b)
        assert n == len(members) and ne == sum(numels[p] for p in members)
        off = 0
        for p in members:
            assert r.param_slot(p) == (b, off)
            off += numels[p]


def test_hand_worked_assignment():
    # fp32, cap 25 MiB: params (MiB) [10, 10, 10, 30, 1] walked from the last:
    # {1, 30} closes at 31 MiB, then {10, 10, 10} closes at 30 MiB.
    mib = MB // 4
    r = Reducer([10 * mib, 10 * mib, 10 * mib, 30 * mib, 1 * mib], B.DP_FP32, K=4,
                bucket_cap_bytes=25 * MB)
    assert r.num_buckets == 2
    assert r.param_slot(4) == (0, 0) and r.param_slot(3) == (0, mib)
    assert r.param_slot(2) == (1, 0) and r.param_slot(1) == (1, 10 * mib)
    assert r.param_slot(0) == (1, 20 * mib)


def test_buckets_launch_in_order_whatever_the_ready_order():
    numels = [1000] * 40
    r = Reducer(numels, B.DP_BF16, K=8, bucket_cap_bytes=2000 * 5)  # 5 params per bucket
    r.set_dry_run(True)
    assert r.num_buckets == 8
    fake = [0x1000 * (k + 1) for k in range(8)]
    for it in range(3):
        order = list(range(40))
        random.Random(it).shuffle(order)
        launched = 0
        for p in order:
            launched += r.mark_ready(p, fake)
        assert launched == 8
        assert r.launch_log() == list(range(8))
        assert r.finish() == (B.DP_OK, -1)


def test_bucket_waits_for_its_last_gradient():
    r = Reducer([10] * 6, B.DP_FP32, K=2, bucket_cap_bytes=80)  # buckets {5,4}, {3,2}, {1,0}
    r.set_dry_run(True)
    fake = [0x100, 0x200]
    assert r.mark_ready(3, fake) == 0  # bucket 1 may not go before bucket 0
    assert r.mark_ready(2, fake) == 0
    assert r.mark_ready(5, fake) == 0
    assert r.mark_ready(4, fake) == 2  # bucket 0 completes; bucket 1 follows at once
    assert r.launch_log() == [0, 1]
    assert r.mark_ready(0, fake) == 0
    assert r.mark_ready(1, fake) == 1
    assert r.finish()[0] == B.DP_OK


def test_unused_parameter_is_reported_not_hung():
    r = Reducer([10] * 6, B.DP_FP32, K=2, bucket_cap_bytes=80)
    r.set_dry_run(True)
    fake = [0x100, 0x200]
    for p in (5, 4, 3, 1, 0):  # parameter 2 takes no part
        r.mark_ready(p, fake)
    st, first_pending = r.finish()
    assert st == B.DP_ERR_INVALID_ARG and first_pending == 1
    # the reducer is reset: a full iteration works again
    for p in range(6):
        r.mark_ready(p, fake)
    assert r.finish() == (B.DP_OK, -1)


def test_double_mark_and_bad_arguments():
    r = Reducer([10] * 4, B.DP_FP32, K=2, bucket_cap_bytes=1 << 20)
    r.set_dry_run(True)
    fake = [0x100, 0x200]
    r.mark_ready(0, fake)
    st, _ = B.dp_reducer_mark_ready(r.handle, 0, fake, stream=0, check=False)
    assert st == B.DP_ERR_INVALID_ARG
    st, _ = B.dp_reducer_mark_ready(r.handle, 9, fake, stream=0, check=False)
    assert st == B.DP_ERR_INVALID_ARG
    st, _ = B.dp_reducer_mark_ready(r.handle, 1, [0x100, None], stream=0, check=False)
    assert st == B.DP_ERR_INVALID_ARG
    st, h = B.dp_reducer_create([10], 1, B.DP_FP32, 0, 100, 1.0, check=False)
    assert st == B.DP_ERR_INVALID_ARG and h == 0
    st, h = B.dp_reducer_create([10], 1, 5, 2, 100, 1.0, check=False)
    assert st == B.DP_ERR_UNSUPPORTED


def test_bucket_allreduce_validation():
    kw = dict(stream=0, check=False)
    base = 0x7F0000000000
    g = [base + i * 4096 for i in range(6)]  # 3 tensors x 2 ranks
    assert B.dp_bucket_allreduce(g, [100, 200, 300], 3, 2, 7, 1.0, **kw) == B.DP_ERR_UNSUPPORTED
    bad = g[:5] + [g[4] + 8]  # overlaps tensor 2 rank 0
    assert B.dp_bucket_allreduce(bad, [100, 200, 300], 3, 2, B.DP_FP32, 1.0, **kw) == 3
    assert B.dp_bucket_allreduce(g[:5] + [None], [1, 1, 1], 3, 2, B.DP_FP32, 1.0, **kw) == 1
    assert B.dp_bucket_allreduce(g, [0, 0, 0], 3, 2, B.DP_FP32, 1.0, **kw) == B.DP_OK


def test_overlap_controls_without_a_device():
    """The overlap mode's host paths: a NULL reducer is rejected; without
    overlap the join has nothing to wait for; switching overlap off when it
    is off is a no-op; switching it on needs a CUDA device, so here it
    reports DP_ERR_CUDA and the reducer keeps working in dry-run mode."""
    import torch
    lib = B.load()
    assert lib.dp_reducer_set_overlap(None, 1) == B.DP_ERR_INVALID_ARG
    assert lib.dp_reducer_wait(None, None) == B.DP_ERR_INVALID_ARG
    red = Reducer([10, 20, 30], B.DP_FP32, 2, bucket_cap_bytes=64, scale=0.5)
    red.set_dry_run(True)
    assert lib.dp_reducer_wait(red.handle, None) == B.DP_OK
    assert lib.dp_reducer_set_overlap(red.handle, 0) == B.DP_OK
    if not torch.cuda.is_available():
        assert lib.dp_reducer_set_overlap(red.handle, 1) == B.DP_ERR_CUDA
    fake = [0x7F0000000000 + i * 4096 for i in range(2)]
    for p in (2, 1, 0):
        red.mark_ready(p, fake)
    assert red.finish() == (B.DP_OK, -1)
