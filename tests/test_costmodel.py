"""Host-side byte accounting, pinned to the worked numbers the pages print."""
import os

import pytest

from ring_allreduce_gradient_gb300 import costmodel as cm

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            out.append(line.split())
    return out


def test_ring_allgather_worked_numbers():
    rows = _rows("ring_cost_worked.txt")
    matrix, shard, W = int(rows[0][0]), int(rows[0][1]), float(rows[0][2]) * 1e9
    assert matrix // 8 == shard
    for X, mb, ms in rows[1:]:
        X = int(X)
        B = shard * X  # completed all-gather buffer: X shards
        sent = cm.ring_allgather_bytes_per_rank(B, X)
        assert sent == shard * (X - 1)
        assert round(sent / 1e6, 3) == pytest.approx(float(mb), abs=5e-4)
        assert round(cm.transport_time_s(sent, W) * 1e3, 2) == pytest.approx(float(ms), abs=5e-3)
        # the reduce-scatter of the matching gradient has the same ideal term
        assert cm.ring_reduce_scatter_bytes_per_rank(B, X) == sent
        assert cm.ring_allreduce_bytes_per_rank(B, X) == 2 * sent


def test_ring_broadcast_terms():
    # whole message: (K-1) N / B; pipelined into S pieces tends to N / B
    assert cm.ring_broadcast_time_s(4, 100.0, 10.0, 1) == pytest.approx(30.0)
    assert cm.ring_broadcast_time_s(4, 100.0, 10.0, 1000) == pytest.approx(10.0 * 1002 / 1000)


def test_hbm_byte_counts():
    MiB = 1 << 20
    # K=8 ranks of 64 Mi bf16, fp32 + bf16 shards: 1 GiB read + 384 MiB written
    assert cm.reduce_scatter_hbm_bytes(8, 64 * MiB, "bf16", ("f32", "bf16")) == 1024 * MiB + 384 * MiB
    assert cm.all_reduce_hbm_bytes(8, 256 * MiB, "f32") == 16 * 1024 * MiB
    assert cm.all_gather_hbm_bytes(8, MiB, "f32") == 8 * MiB * 4 * 9
    assert cm.gemm_flops(8192, 4096, 4096) == 274877906944
    assert cm.accumulate_hbm_bytes(10, "bf16", first=True) == 60
    assert cm.accumulate_hbm_bytes(10, "bf16", first=False) == 100
    assert cm.accumulate_hbm_bytes(10, "bf16", first=False, pad=True) == 80
