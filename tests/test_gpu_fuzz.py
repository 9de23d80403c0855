"""GPU parity under a seeded random mix: sequences of collective calls with
random rank counts, sizes (ragged included), dtypes, 16-byte and odd view
offsets, implementation variants and streaming CTA caps, launched round-robin
on three streams so that independent calls run at the same time, then every
result compared bit for bit with the oracle.  Each case owns its buffers."""
import random

import numpy as np
import pytest
import torch

import oracle
import workloads
from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import collectives as col

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def host_ranks(rng, K, N, dt):
    f = [rng.uniform(-1, 1, N).astype(np.float32) for _ in range(K)]
    return [workloads.to_bf16_bits(a) for a in f] if dt == "bf16" else f


def to_dev(a, offset):
    """A device copy of `a` starting `offset` elements into its allocation."""
    t = workloads.bits_to_torch_bf16(a) if a.dtype == np.uint16 else torch.from_numpy(a)
    raw = torch.empty(a.size + offset, dtype=t.dtype, device=DEV)
    raw[offset:].copy_(t)
    return raw[offset:]


def empty(n, tdt, offset):
    return torch.empty(n + offset, dtype=tdt, device=DEV)[offset:]


def bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


def as_bits(a):
    return a.view(np.int16) if a.dtype == np.uint16 else a.view(np.int32)


TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def case_rs(rng, s):
    K = int(rng.integers(1, 17))
    dt = ["f32", "bf16"][rng.integers(2)]
    C = int(rng.choice([1, 7, 8, 1000, 4099, 8 * 3001]))
    off = int(rng.choice([0, 0, 4 if dt == "f32" else 8, 1]))
    host = host_ranks(rng, K, K * C, dt)
    bufs = [to_dev(h, off) for h in host]
    o32 = [empty(C, torch.float32, off) for _ in range(K)]
    o16 = [empty(C, torch.bfloat16, off) for _ in range(K)]
    scale = float(rng.choice([1.0, 1.0 / K, -0.5]))
    B.dp_reduce_scatter_dual(bufs, K, K * C, TDT[dt], o32, o16, scale, s)

    def check():
        r32, r16 = oracle.reduce_scatter(host, scale)
        for c in range(K):
            assert np.array_equal(bits(o32[c]), as_bits(r32[c])), ("rs32", K, dt, C, off, c)
            assert np.array_equal(bits(o16[c]), as_bits(r16[c])), ("rs16", K, dt, C, off, c)
    return check, (bufs, o32, o16)


def case_ag(rng, s):
    K = int(rng.integers(1, 17))
    dt = ["f32", "bf16"][rng.integers(2)]
    C = int(rng.choice([4, 8, 1000, 16384 + 4, 3 * 16384]))
    off = int(rng.choice([0, 0, 4 if dt == "f32" else 8, 1]))
    host = host_ranks(rng, K, C, dt)
    shards = [to_dev(h, off) for h in host]
    out = [empty(K * C, TDT[dt], off) for _ in range(K)]
    if rng.integers(4) == 0:
        B.dp_all_gather_copy_engine(shards, K, C, TDT[dt], out, s)
    else:
        B.dp_all_gather(shards, K, C, TDT[dt], out, s)

    def check():
        ref = oracle.all_gather(host)
        for r in range(K):
            assert np.array_equal(bits(out[r]), as_bits(ref[r])), ("ag", K, dt, C, off, r)
    return check, (shards, out)


def case_ar(rng, s):
    K = int(rng.integers(1, 17))
    dt = ["f32", "bf16"][rng.integers(2)]
    N = int(rng.choice([1, 13, 4096, 8 * 5000 + 3, 65536 * 3]))
    off = int(rng.choice([0, 0, 4 if dt == "f32" else 8, 1]))
    host = host_ranks(rng, K, N, dt)
    bufs = [to_dev(h, off) for h in host]
    scale = float(rng.choice([1.0, 1.0 / K]))
    B.dp_ring_allreduce(bufs, K, N, TDT[dt], scale, s)

    def check():
        ref = oracle.all_reduce(host, scale)
        for r in range(K):
            assert np.array_equal(bits(bufs[r]), as_bits(ref[r])), ("ar", K, dt, N, off, r)
    return check, (bufs,)


def case_bucket(rng, s):
    K = int(rng.integers(1, 9))
    dt = ["f32", "bf16"][rng.integers(2)]
    sizes = [int(rng.choice([1, 5, 8, 100, 4099, 65536])) for _ in range(rng.integers(1, 7))]
    host = [host_ranks(rng, 1, n, dt)[0] for n in sizes for _ in range(K)]
    host = [[host[i * K + r] for i in range(len(sizes))] for r in range(K)]
    dev = [[to_dev(a, 0) for a in row] for row in host]
    scale = 1.0 / K
    grads = [dev[r][t] for t in range(len(sizes)) for r in range(K)]
    B.dp_bucket_allreduce(grads, sizes, len(sizes), K, TDT[dt], scale, s)

    def check():
        ref = oracle.bucket_all_reduce(host, scale)
        for r in range(K):
            for i in range(len(sizes)):
                assert np.array_equal(bits(dev[r][i]), as_bits(ref[r][i])), ("bucket", K, i)
    return check, (dev,)


def case_odc(rng, s):
    K = int(rng.integers(1, 9))
    C = int(rng.choice([8, 1000, 8 * 777]))
    N = K * C
    m = [int(rng.integers(0, 4)) for _ in range(K)]
    hg = [[workloads.to_bf16_bits(rng.standard_normal(N).astype(np.float32) * np.float32(1e-3))
           for _ in range(m[r])] for r in range(K)]
    dg = [[to_dev(g, 0) for g in row] for row in hg]
    o32, o16 = col.odc_reduce_scatter(dg, m, N, 1.0 / K, device=DEV, stream=s)

    def check():
        e32, e16 = oracle.odc_layer(hg, m, 1.0 / K, N)
        for c in range(K):
            assert np.array_equal(bits(o32[c]), as_bits(e32[c])), ("odc32", K, C, m, c)
            assert np.array_equal(bits(o16[c]), as_bits(e16[c])), ("odc16", K, C, m, c)
    return check, (dg, o32, o16)


def case_pipe(rng, s):
    """A layer settled in microbatch groups through a settle pipe (its own
    side stream, forked from and joined back to `s`)."""
    K = int(rng.integers(1, 9))
    C = int(rng.choice([8, 1000, 8 * 777]))
    N = K * C
    m = [int(rng.integers(1, 6)) for _ in range(K)]
    M = max(m)
    cut = sorted({0, M} | {int(v) for v in rng.integers(1, M + 1, size=int(rng.integers(0, 3)))})
    hg = [[workloads.to_bf16_bits(rng.standard_normal(N).astype(np.float32) * np.float32(1e-3))
           for _ in range(m[r])] for r in range(K)]
    dg = [[to_dev(g, 0) for g in row] for row in hg]
    pipe = col.SettlePipe(K, N, DEV, cta_limit=int(rng.choice([0, 0, 16])))
    G = len(cut) - 1
    for g, (lo, hi) in enumerate(zip(cut[:-1], cut[1:])):
        pipe.push([row[lo:hi] for row in dg], first=(g == 0), last=(g == G - 1),
                  scale=1.0 / K, stream=s)
    pipe.wait(stream=s)

    def check():
        e32, e16 = oracle.odc_pipelined(hg, m, cut, 1.0 / K, N)
        for c in range(K):
            assert np.array_equal(bits(pipe.out32[c]), as_bits(e32[c])), ("pipe32", K, C, m, cut)
            assert np.array_equal(bits(pipe.out16[c]), as_bits(e16[c])), ("pipe16", K, C, m, cut)
        pipe.close()
    return check, (dg, pipe)


def case_reducer(rng, s):
    """One DDP iteration of a Reducer in overlap mode (buckets on its two
    streams), joined back to `s`."""
    from tests.test_reducer_cpu import expected_buckets
    K = int(rng.integers(1, 9))
    numels = [int(rng.choice([1, 7, 64, 1000, 4099, 65536])) for _ in range(rng.integers(1, 12))]
    cap = int(rng.choice([256, 16384, 1 << 20]))
    host = [[host_ranks(rng, 1, n, "f32")[0] for n in numels] for _ in range(K)]
    dev = [[to_dev(a, 0) for a in row] for row in host]
    red = col.Reducer(numels, B.DP_FP32, K, bucket_cap_bytes=cap, scale=1.0 / K)
    red.set_overlap(True)
    for p in reversed(range(len(numels))):
        red.mark_ready(p, [dev[r][p] for r in range(K)], stream=s)
    red.wait(stream=s)
    assert red.finish() == (B.DP_OK, -1)

    def check():
        for members in expected_buckets(numels, 4, cap):
            ref = oracle.bucket_all_reduce([[host[r][q] for q in members] for r in range(K)],
                                           1.0 / K)
            for r in range(K):
                for i, q in enumerate(members):
                    assert np.array_equal(bits(dev[r][q]), as_bits(ref[r][i])), ("reducer", q, r)
        red.set_overlap(False)
    return check, (dev, red)


CASES = [case_rs, case_ag, case_ar, case_bucket, case_odc, case_pipe, case_reducer]


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5, 6])
def test_random_mix_on_three_streams(seed):
    rng = np.random.default_rng(1000 + seed)
    pick = random.Random(seed)
    streams = [torch.cuda.Stream() for _ in range(3)]
    saved_variant = B.dp_get_collective_variant()
    saved_limits = B.dp_get_cta_limits()
    checks, keep = [], []
    torch.cuda.synchronize()
    try:
        for i in range(32):
            B.dp_set_collective_variant(pick.choice([0, 0, 1, 2]))
            B.dp_set_cta_limits(saved_limits[0], pick.choice([0, 0, 0, 8, 40, 100]))
            s = streams[i % 3]
            with torch.cuda.stream(s):
                chk, k = pick.choice(CASES)(rng, s.cuda_stream)
            checks.append(chk)
            keep.append(k)
        torch.cuda.synchronize()
    finally:
        B.dp_set_collective_variant(saved_variant)
        B.dp_set_cta_limits(*saved_limits)
    assert B.dp_get_device_error() == B.DP_OK
    for chk in checks:
        chk()


# ---------------------------------------------------------------------------
# tensor-core calls: random shapes, integer operands (every fp32 sum exact, so
# the results equal the fp64 oracle), random GEMM CTA caps (which make the
# chained split of a part-full last round appear), with and without a
# workspace (bitwise the same)
# ---------------------------------------------------------------------------

def _i(rng, choices):
    return int(rng.choice(choices))


def gemm_gather(rng):
    K, M, D, Fs = _i(rng, [1, 2, 3, 8]), _i(rng, [1, 77, 128, 300]), _i(rng, [8, 64, 200, 256]), \
        _i(rng, [16, 48, 64])
    x, ws = workloads.gemm_int_operands(M, D, K, Fs, seed=int(rng.integers(1 << 30)))
    xd = workloads.bits_to_torch_bf16(x).to(DEV)
    wd = [workloads.bits_to_torch_bf16(w).to(DEV) for w in ws]
    run = lambda wsp: [col.allgather_matmul(xd, wd, torch.float32, workspace=wsp)]
    ref = lambda: [oracle.allgather_matmul_f64(x, ws)]
    return run, ref, ("gather", K, M, D, Fs)


def gemm_tp(rng):
    K = _i(rng, [1, 2, 4, 8])
    M, Ds = K * _i(rng, [16, 50, 64]), _i(rng, [8, 64, 128])
    xw = bool(rng.integers(2))
    F = _i(rng, [64, 128, 192]) if xw else _i(rng, [16, 48, 64, 160])
    scatter = bool(rng.integers(2))
    xs, ws = workloads.tp_operands(M, Ds, F, K, ints=True)
    xd = [workloads.bits_to_torch_bf16(a).to(DEV) for a in xs]
    wd = [workloads.bits_to_torch_bf16(np.ascontiguousarray(w.T) if xw else w).to(DEV)
          for w in ws]
    fn = {(False, False): col.matmul_allreduce, (False, True): col.matmul_reduce_scatter,
          (True, False): col.matmul_allreduce_xw, (True, True): col.matmul_reduce_scatter_xw}
    run = lambda wsp: fn[(xw, scatter)](xd, wd, 0.5, torch.float32, workspace=wsp)

    def ref():
        y = oracle.matmul_psum_f64(xs, ws, 0.5)
        return np.split(y, K, axis=0) if scatter else [y] * K
    return run, ref, ("tp", K, M, Ds, F, xw, scatter)


def gemm_wgrad(rng):
    K = _i(rng, [1, 2, 4, 8])
    T, F, D = _i(rng, [1, 64, 200]), 64 * _i(rng, [1, 2, 4]), 64 * _i(rng, [1, 3])
    dys, xs = workloads.wgrad_operands(T, F, D, K, ints=True)
    dd = [workloads.bits_to_torch_bf16(a).to(DEV) for a in dys]
    xd = [workloads.bits_to_torch_bf16(a).to(DEV) for a in xs]
    run = lambda wsp: col.wgrad_reduce_scatter(dd, xd, 0.25, torch.float32, workspace=wsp)
    ref = lambda: np.split(oracle.wgrad_psum_f64(dys, xs, 0.25), K, axis=0)
    return run, ref, ("wgrad", K, T, F, D)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_gemms_under_random_cta_caps(seed):
    rng = np.random.default_rng(2000 + seed)
    saved = B.dp_get_cta_limits()
    try:
        for _ in range(12):
            run, ref, tag = [gemm_gather, gemm_tp, gemm_wgrad][int(rng.integers(3))](rng)
            B.dp_set_cta_limits(_i(rng, [0, 0, 3, 5, 15, 40]), saved[1])
            with_ws = run("auto")
            without = run(None)
            torch.cuda.synchronize()
            assert B.dp_get_device_error() == B.DP_OK, tag
            want = ref()
            for a, b, w in zip(with_ws, without, want):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32)), tag
                assert np.array_equal(a.cpu().numpy().astype(np.float64), w), tag
    finally:
        B.dp_set_cta_limits(*saved)
