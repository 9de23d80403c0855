"""GPU parity of the variable-length microbatch step: per-rank accumulation
(dp_grad_accumulate) and the fused accumulate + settle (dp_odc_reduce_scatter),
padded and unpadded, bit for bit against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def f32bits(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def host_grads(K, N, m, seed, dt="bf16"):
    rng = np.random.default_rng(seed)
    out = []
    for r in range(K):
        row = []
        for j in range(m[r]):
            g = rng.standard_normal(N).astype(np.float32) * np.float32(1e-3 * (1 + j))
            row.append(workloads.to_bf16_bits(g) if dt == "bf16" else g)
        out.append(row)
    return out


def to_dev(a):
    if a.dtype == np.uint16:
        return workloads.bits_to_torch_bf16(a).to(DEV)
    return torch.from_numpy(a).to(DEV)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("N", [8 * 8 * 1500, 8 * 1001])
def test_fused_step_padded_equals_unpadded_equals_oracle(dt, N):
    K = 8
    m, _ = workloads.odc_schedule(K)
    hg = host_grads(K, N, m, 21, dt)
    dg = [[to_dev(g) for g in row] for row in hg]
    gdt = torch.bfloat16 if dt == "bf16" else torch.float32
    a32, a16 = col.odc_reduce_scatter(dg, m, N, 1.0 / K, gdt)
    M = max(m)
    padded = [row + [None] * (M - len(row)) for row in dg]
    b32, b16 = col.odc_reduce_scatter(padded, [M] * K, N, 1.0 / K, gdt)
    e32, e16 = oracle.odc_layer(hg, m, 1.0 / K, N, grad_dtype=1 if dt == "bf16" else 0)
    for c in range(K):
        assert np.array_equal(f32bits(a32[c]), e32[c].view(np.uint32))
        assert np.array_equal(f32bits(b32[c]), e32[c].view(np.uint32))
        assert np.array_equal(workloads.torch_bf16_to_bits(a16[c]), e16[c])
        assert np.array_equal(workloads.torch_bf16_to_bits(b16[c]), e16[c])


@pytest.mark.parametrize("K,m,holes,dt,N", [
    # ranks without microbatches (one right after a chunk's owner, where the
    # ring-ordered list of that chunk starts), padding inside a rank's list
    # and at its start
    (8, [0, 3, 0, 1, 4, 2, 0, 5], {(1, 1), (4, 0)}, "bf16", 8 * 8 * 1000),
    (3, [2, 0, 1], set(), "f32", 3 * 8 * 999),
    (16, [1, 0, 0, 2] * 4, {(3, 0), (15, 1)}, "bf16", 16 * 8 * 300),
    # chunk length not a multiple of 8: the scalar kernel, same schedule
    (8, [0, 3, 0, 1, 4, 2, 0, 5], {(1, 1), (4, 0)}, "bf16", 8 * 1001),
])
def test_fused_step_empty_ranks_and_padding_inside(K, m, holes, dt, N):
    hg = host_grads(K, N, m, 31, dt)
    for r, j in holes:
        hg[r][j] = None
    dg = [[None if g is None else to_dev(g) for g in row] for row in hg]
    gdt = torch.bfloat16 if dt == "bf16" else torch.float32
    a32, a16 = col.odc_reduce_scatter(dg, m, N, 1.0 / K, gdt, device=DEV)
    e32, e16 = oracle.odc_layer(hg, m, 1.0 / K, N, grad_dtype=1 if dt == "bf16" else 0)
    for c in range(K):
        assert np.array_equal(f32bits(a32[c]), e32[c].view(np.uint32))
        assert np.array_equal(workloads.torch_bf16_to_bits(a16[c]), e16[c])


def test_fused_step_of_padding_only_is_positive_zero():
    K, N = 8, 8 * 8 * 64
    grads = [[None, None] for _ in range(K)]
    a32, a16 = col.odc_reduce_scatter(grads, [2] * K, N, 1.0 / K, torch.bfloat16, device=DEV)
    for c in range(K):
        assert not f32bits(a32[c]).any()  # +0 everywhere (no -0)
        assert not workloads.torch_bf16_to_bits(a16[c]).any()


def test_two_phase_path_equals_fused_and_oracle():
    """Accumulate each microbatch into an fp32 buffer per rank (padding
    buckets included), then settle with the reduce-scatter: identical bits."""
    K, N = 8, 8 * 8 * 700 + 8 * 3
    m = [2, 1, 4, 3, 1, 5, 2, 3]
    M = max(m)
    hg = host_grads(K, N, m, 22)
    dg = [[to_dev(g) for g in row] for row in hg]
    accs = [torch.full((N,), 12345.0, device=DEV) for _ in range(K)]
    for r in range(K):
        for j in range(M):  # padded run: ranks with m[r] < M add padding buckets
            g = dg[r][j] if j < m[r] else None
            col.grad_accumulate_(accs[r], g, first=(j == 0))
    s32, s16 = col.reduce_scatter(accs, 1.0 / K)
    f32_, f16_ = col.odc_reduce_scatter(dg, m, N, 1.0 / K)
    e32, e16 = oracle.odc_layer(hg, m, 1.0 / K, N)
    for c in range(K):
        assert np.array_equal(f32bits(s32[c]), e32[c].view(np.uint32))
        assert np.array_equal(f32bits(f32_[c]), e32[c].view(np.uint32))
        assert np.array_equal(workloads.torch_bf16_to_bits(s16[c]), e16[c])


@pytest.mark.parametrize("first", [True, False])
@pytest.mark.parametrize("pad", [True, False])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("N,off", [(8 * 4099, 0), (8 * 4099 + 5, 0), (1003, 1)])
def test_accumulate_matches_oracle(first, pad, dt, N, off):
    rng = np.random.default_rng(N + off)
    acc0 = rng.standard_normal(N).astype(np.float32)
    g = rng.standard_normal(N).astype(np.float32)
    g = workloads.to_bf16_bits(g) if dt == "bf16" else g
    raw = torch.empty(N + off, device=DEV)
    acc = raw[off:]
    acc.copy_(torch.from_numpy(acc0))
    graw = None
    if not pad:
        gt = to_dev(g)
        graw = torch.empty(N + off, dtype=gt.dtype, device=DEV)
        graw[off:].copy_(gt)
    gdt = B.DP_BF16 if dt == "bf16" else B.DP_FP32
    B.dp_grad_accumulate(acc, None if pad else graw[off:], N, gdt, first)
    want = acc0.copy()
    oracle.accumulate(want, None if pad else g, first)
    assert np.array_equal(f32bits(acc), want.view(np.uint32))


def test_full_layer_sampled():
    """One layer of the variable-length step at full size: K=8, 16 Mi
    elements, microbatch counts and token scales from the schedule, gradients
    drawn on the device; sampled elements against the oracle."""
    K, N = 8, 16 * workloads.MiB
    C = N // K
    m, toks = workloads.odc_schedule(K)
    layer = 3
    dg = [[workloads.odc_grad(layer, r, j, N, int(toks[r, j]), DEV) for j in range(m[r])]
          for r in range(K)]
    o32, o16 = col.odc_reduce_scatter(dg, m, N, 1.0 / K)
    M = max(m)
    p32, _ = col.odc_reduce_scatter([row + [None] * (M - len(row)) for row in dg], [M] * K, N,
                                    1.0 / K)
    for c in range(K):
        assert torch.equal(o32[c].view(torch.int32), p32[c].view(torch.int32))
    rng = np.random.default_rng(4)
    idx = np.unique(np.concatenate([rng.integers(0, N, 1024), [0, C - 1, C, N - 1]]))
    it = torch.from_numpy(idx).to(DEV)
    S = idx.size
    small = []
    for r in range(K):
        row = []
        for j in range(m[r]):
            v = workloads.torch_bf16_to_bits(dg[r][j][it])
            buf = np.zeros(K * S, np.uint16)
            buf[(idx // C) * S + np.arange(S)] = v
            row.append(buf)
        small.append(row)
    e32, e16 = oracle.odc_layer(small, m, 1.0 / K, K * S)
    got = np.stack([f32bits(o32[c]) for c in range(K)])
    for s, e in enumerate(idx):
        c, i = divmod(int(e), C)
        assert got[c, i] == e32[c][s].view(np.uint32)


def _golden_odc(name):
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    K, N = map(int, rows[0].split())
    per_rank = [[float(v) for v in rows[1 + r].split()] for r in range(K)]
    return K, N, per_rank, rows[1 + K:]


@pytest.mark.parametrize("rep", [1, 1024])
def test_association_by_hand_fused_and_two_phase(rep):
    """The hand-worked binary32 values of the microbatch association pin
    (per-rank ascending accumulation, then one ring settle), on the GPU: the
    fused kernel (scalar path at the pin's size, vector path when every chunk
    is repeated 1024 times) and the two-phase path both give them."""
    K, N0, per_rank, rest = _golden_odc("odc_association_k2.txt")
    expect = [float(v) for v in rest[0].split()]
    N = N0 * rep
    m = [len(v) for v in per_rank]
    dg = [[torch.full((N,), v, dtype=torch.bfloat16, device=DEV) for v in vals]
          for vals in per_rank]
    a32, a16 = col.odc_reduce_scatter(dg, m, N, 1.0)
    accs = [torch.empty(N, device=DEV) for _ in range(K)]
    for r in range(K):
        for j, g in enumerate(dg[r]):
            col.grad_accumulate_(accs[r], g, first=(j == 0))
    s32, _ = col.reduce_scatter(accs, 1.0)
    for c in range(K):
        want = torch.full((N // K,), expect[c])
        assert torch.equal(a32[c].cpu(), want)
        assert torch.equal(a16[c].float().cpu(), want)
        assert torch.equal(s32[c].cpu(), want)
