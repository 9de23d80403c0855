"""Pins for the CPU oracle: it is checked here against facts that do not come
from itself -- the pages' ring walk, hand-worked binary32 values, brute-force
exact sums, closed forms, error bounds and independent library routines
(PyTorch's bf16 conversion, numpy's float64 matmul and concatenate).

Every check is a plain function taking no arguments so that
``test_oracle_mutants.py`` can re-run the whole set against an oracle with a
planted mistake and show that at least one of them fails.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


def _bits(a):
    return np.asarray(a).view(np.uint32) if np.asarray(a).dtype == np.float32 else np.asarray(a)


# --------------------------------------------------------------------------
# bf16 conversions: against PyTorch's own conversion (an independent library)
# --------------------------------------------------------------------------

def pin_bf16_round_matches_torch():
    rng = np.random.default_rng(123)
    vals = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(1e-3),
        rng.uniform(-1e30, 1e30, 500).astype(np.float32),
        # exact ties and near-ties around 1.0 and 2^-130 (subnormal range)
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8),
                  2.0 ** -130, 3 * 2.0 ** -140, 0.0, -0.0, np.inf, -np.inf,
                  3.3895314e38, 3.4028235e38, -3.4028235e38], dtype=np.float32),
        (rng.integers(0, 2 ** 32, 2000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
    ])
    vals = vals[~np.isnan(vals)]
    ours = oracle.bf16_round(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def pin_bf16_ties_by_hand():
    # 1 + 2^-8 is halfway between 1.0 and 1.0078125: the even one is 1.0.
    # 1 + 3*2^-8 is halfway between 1.0078125 and 1.015625: even is 1.015625.
    got = oracle.bf16_widen(oracle.bf16_round(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8],
                                                       dtype=np.float32)))
    assert got.tolist() == [1.0, 1.015625]
    nan = oracle.bf16_widen(oracle.bf16_round(np.array([np.nan], np.float32)))
    assert np.isnan(nan[0])


def pin_bf16_widen_all_patterns():
    pats = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_widen(pats)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


# --------------------------------------------------------------------------
# The pages' ring walk and hand-worked pins
# --------------------------------------------------------------------------

def pin_symbolic_ring_walk():
    rows = _golden_rows("ring_walk_k4.txt")
    K, N = map(int, rows[0].split())
    labels = [float(v) for v in rows[1].split()]
    expect = {int(a): float(b) for a, b in (r.split(":") for r in rows[2:])}
    bufs = [np.full(N, labels[w], np.float32) for w in range(K)]
    f32, _ = oracle.reduce_scatter(bufs, 1.0, ("f32",))
    for c in range(K):
        assert np.all(f32[c] == expect[c]), (c, f32[c])
    ar = oracle.all_reduce(bufs, 1.0)
    for r in range(K):
        assert np.all(ar[r] == 15.0)


def pin_ring_rotation():
    rows = _golden_rows("ring_rotation_k4.txt")
    K, N = map(int, rows[0].split())
    per_rank = [float(v) for v in rows[1].split()]
    expect = [float(v) for v in rows[2].split()]
    bufs = [np.full(N, per_rank[r], np.float32) for r in range(K)]
    f32, _ = oracle.reduce_scatter(bufs, 1.0, ("f32",))
    assert [float(s[0]) for s in f32] == expect
    fold, _ = oracle.reduce_scatter_fold(bufs, 1.0, ("f32",))
    assert [float(s[0]) for s in fold] == expect
    ar = oracle.all_reduce(bufs, 1.0)
    C = N // K
    for r in range(K):
        assert [float(ar[r][c * C]) for c in range(K)] == expect


# --------------------------------------------------------------------------
# Brute force on integer-valued inputs (every order is exact)
# --------------------------------------------------------------------------

def pin_config1_bruteforce():
    bufs = workloads.ring_ints(K=4, N=4096, seed=0)
    exact = [sum(int(b[e]) for b in bufs) for e in range(4096)]
    f32, b16 = oracle.reduce_scatter(bufs, 1.0)
    C = 1024
    for c in range(4):
        assert f32[c].tolist() == [float(v) for v in exact[c * C:(c + 1) * C]]
        assert oracle.bf16_widen(b16[c]).tolist() == [float(v) for v in exact[c * C:(c + 1) * C]]
    ar = oracle.all_reduce(bufs, 1.0)
    for r in range(4):
        assert ar[r].tolist() == [float(v) for v in exact]


def pin_integer_ragged_allreduce():
    # N % K != 0: chunks of ceil(N/K), the last ones short or empty
    for K, N in [(3, 10), (4, 5), (8, 9), (5, 3), (7, 1)]:
        rng = np.random.default_rng(K * 100 + N)
        bufs = [rng.integers(-8, 9, N).astype(np.float32) for _ in range(K)]
        exact = np.sum(np.stack(bufs).astype(np.int64), axis=0).astype(np.float32)
        for out in oracle.all_reduce(bufs, 1.0):
            assert np.array_equal(out, exact)


# --------------------------------------------------------------------------
# Closed forms and invariants
# --------------------------------------------------------------------------

def _rand_bufs(K, N, dtype, seed):
    rng = np.random.default_rng(seed)
    f = [rng.uniform(-1, 1, N).astype(np.float32) for _ in range(K)]
    if dtype == "bf16":
        return [workloads.to_bf16_bits(a) for a in f]
    return f


def pin_sim_equals_closed_form():
    for K in range(1, 9):
        for dt in ("f32", "bf16"):
            N = K * 37
            bufs = _rand_bufs(K, N, dt, 10 * K)
            for scale in (1.0, 1.0 / K, 0.3):
                a32, a16 = oracle.reduce_scatter(bufs, scale)
                b32, b16 = oracle.reduce_scatter_fold(bufs, scale)
                for c in range(K):
                    assert np.array_equal(_bits(a32[c]), _bits(b32[c]))
                    assert np.array_equal(a16[c], b16[c])


def pin_fold_within_recursive_sum_bound():
    # |fl(sum) - sum| <= gamma_{K-1} * sum |x_i|, gamma_n = n u / (1 - n u),
    # u = 2^-24 (recursive summation error bound), and the fp32 fold must not
    # be exact-by-accident on this data (it differs from fp64 somewhere).
    u = 2.0 ** -24
    for K in (2, 4, 8, 16):
        N = K * 500
        bufs = _rand_bufs(K, N, "f32", 77 + K)
        f32, _ = oracle.reduce_scatter(bufs, 1.0, ("f32",))
        got = np.concatenate(f32).astype(np.float64)
        X = np.stack(bufs).astype(np.float64)
        exact = X.sum(axis=0)
        gamma = (K - 1) * u / (1 - (K - 1) * u)
        assert np.all(np.abs(got - exact) <= gamma * np.abs(X).sum(axis=0) + 1e-300)
        if K > 2:
            assert np.any(got != exact)


def pin_k2_is_one_library_add():
    # K = 2: shard c = x_{c+1} + x_c, one IEEE fp32 add (numpy's)
    bufs = _rand_bufs(2, 2 * 301, "f32", 5)
    f32, _ = oracle.reduce_scatter(bufs, 1.0, ("f32",))
    C = 301
    np_sum = (bufs[1] + bufs[0]).astype(np.float32)
    assert np.array_equal(np.concatenate(f32), np_sum)
    assert C == f32[0].size


def pin_allreduce_is_rs_then_ag():
    for K in (1, 2, 3, 4, 8):
        for dt in ("f32", "bf16"):
            N = K * 64
            bufs = _rand_bufs(K, N, dt, 900 + K)
            scale = 1.0 / K
            ar = oracle.all_reduce(bufs, scale)
            f32, b16 = oracle.reduce_scatter(bufs, scale)
            shards = f32 if dt == "f32" else b16
            ag = oracle.all_gather(shards)
            for r in range(K):
                assert np.array_equal(_bits(ar[r]), _bits(ag[r]))
                assert np.array_equal(_bits(ar[r]), _bits(ar[0]))  # every rank identical


def pin_ragged_allreduce_matches_padded():
    # The all-reduce of a ragged N equals the divisible case on the buffer
    # padded to K*ceil(N/K): an element's result depends only on its chunk.
    for K, N in [(3, 10), (4, 13), (8, 60), (8, 3)]:
        bufs = _rand_bufs(K, N, "f32", K + N)
        C = -(-N // K)
        padded = [np.concatenate([b, np.zeros(K * C - N, np.float32)]) for b in bufs]
        ar = oracle.all_reduce(bufs, 1.0 / K)
        f32, _ = oracle.reduce_scatter(padded, 1.0 / K, ("f32",))
        full = np.concatenate(f32)[:N]
        for r in range(K):
            assert np.array_equal(_bits(ar[r]), _bits(full))


def pin_k1_special_case():
    x = _rand_bufs(1, 97, "f32", 3)
    f32, b16 = oracle.reduce_scatter(x, 0.5)
    assert np.array_equal(f32[0], x[0] * np.float32(0.5))
    assert np.array_equal(b16[0], workloads.to_bf16_bits(x[0] * np.float32(0.5)))
    assert np.array_equal(oracle.all_gather(x)[0], x[0])


def pin_power_of_two_scale_commutes():
    # fold(x) * 2^-k == fold(x * 2^-k) bit for bit (no under/overflow here)
    for K in (2, 4, 8):
        bufs = _rand_bufs(K, K * 50, "f32", 40 + K)
        a, _ = oracle.reduce_scatter(bufs, 2.0 ** -3, ("f32",))
        scaled = [b * np.float32(2.0 ** -3) for b in bufs]
        b, _ = oracle.reduce_scatter(scaled, 1.0, ("f32",))
        for c in range(K):
            assert np.array_equal(_bits(a[c]), _bits(b[c]))


def pin_scale_is_applied():
    bufs = workloads.ring_ints(K=4, N=64, seed=1)
    f32, _ = oracle.reduce_scatter(bufs, 0.25, ("f32",))
    exact = np.sum(np.stack(bufs), axis=0) / 4.0
    assert np.array_equal(np.concatenate(f32), exact.astype(np.float32))


def pin_all_gather_is_concatenation():
    for K in (1, 2, 5, 8):
        for dt in (np.float32, np.uint16):
            rng = np.random.default_rng(K)
            shards = [rng.integers(0, 60000, 33).astype(dt) for _ in range(K)]
            cat = np.concatenate(shards)
            for out in oracle.all_gather(shards):
                assert np.array_equal(out, cat)


def pin_bf16_output_is_rounded_fp32_output():
    bufs = _rand_bufs(8, 8 * 128, "bf16", 8)
    f32, b16 = oracle.reduce_scatter(bufs, 1.0 / 8)
    for c in range(8):
        ref = torch.from_numpy(f32[c]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(b16[c], ref)


# --------------------------------------------------------------------------
# FSDP all-gather + local GEMM (fp64 reference)
# --------------------------------------------------------------------------

def pin_gemm_bruteforce_tiny():
    x, ws = workloads.gemm_operands(M=5, D=7, K=3, F_shard=2)
    y = oracle.allgather_matmul_f64(x, ws)
    xf = oracle.bf16_widen(x).astype(np.float64)
    w = [oracle.bf16_widen(s).astype(np.float64) for s in ws]
    for m in range(5):
        for k in range(3):
            for f in range(2):
                acc = 0.0
                for d in range(7):
                    acc += float(xf[m, d]) * float(w[k][f, d])
                assert y[m, k * 2 + f] == acc


def pin_gemm_matches_numpy_f64():
    x, ws = workloads.gemm_operands(M=64, D=96, K=4, F_shard=16)
    y = oracle.allgather_matmul_f64(x, ws)
    xf = oracle.bf16_widen(x).astype(np.float64)
    wf = np.concatenate([oracle.bf16_widen(s).astype(np.float64) for s in ws])
    ref = xf @ wf.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)


def pin_gemm_integer_exact():
    x, ws = workloads.gemm_int_operands(M=32, D=128, K=4, F_shard=16, seed=3)
    y = oracle.allgather_matmul_f64(x, ws)
    xi = oracle.bf16_widen(x).astype(np.int64)
    wi = np.concatenate([oracle.bf16_widen(s).astype(np.int64) for s in ws])
    assert np.array_equal(y, (xi @ wi.T).astype(np.float64))


def pin_gemm_square_orientation():
    # w square: x . w^T and x . w differ, so a transposed operand is caught
    x, ws = workloads.gemm_operands(M=8, D=32, K=4, F_shard=8)
    y = oracle.allgather_matmul_f64(x, ws)
    xf = oracle.bf16_widen(x).astype(np.float64)
    wf = np.concatenate([oracle.bf16_widen(s).astype(np.float64) for s in ws])
    assert np.allclose(y, xf @ wf.T, rtol=1e-12, atol=1e-15)


def pin_gemm_sampled_equals_full():
    x, ws = workloads.gemm_operands(M=16, D=64, K=2, F_shard=8)
    y = oracle.allgather_matmul_f64(x, ws)
    ms = np.array([0, 3, 15, 7], np.int64)
    fs = np.array([0, 9, 15, 8], np.int64)
    assert np.array_equal(oracle.allgather_matmul_f64_sampled(x, ws, ms, fs), y[ms, fs])


# --------------------------------------------------------------------------
# Tensor-parallel psum of partial dots (fp64 reference)
# --------------------------------------------------------------------------

def pin_psum_equals_unsharded_product():
    # splitting the contracted dimension over the ranks and summing the
    # partial dots is the unsharded product x . w^T (numpy fp64 matmul)
    xs, ws = workloads.tp_operands(M=24, D_shard=16, F=20, K=4)
    y = oracle.matmul_psum_f64(xs, ws)
    x = np.concatenate([oracle.bf16_widen(a).astype(np.float64) for a in xs], axis=1)
    w = np.concatenate([oracle.bf16_widen(b).astype(np.float64) for b in ws], axis=1)
    assert np.allclose(y, x @ w.T, rtol=1e-12, atol=1e-15)


def pin_psum_integer_exact_and_scaled():
    xs, ws = workloads.tp_operands(M=16, D_shard=32, F=16, K=8, ints=True)
    y = oracle.matmul_psum_f64(xs, ws, scale=0.125)
    x = np.concatenate([oracle.bf16_widen(a).astype(np.int64) for a in xs], axis=1)
    w = np.concatenate([oracle.bf16_widen(b).astype(np.int64) for b in ws], axis=1)
    assert np.array_equal(y, (x @ w.T).astype(np.float64) * 0.125)


def pin_psum_one_rank_is_the_plain_gemm():
    xs, ws = workloads.tp_operands(M=12, D_shard=40, F=24, K=1)
    y = oracle.matmul_psum_f64(xs, ws)
    assert np.array_equal(y, oracle.allgather_matmul_f64(xs[0], ws))


def pin_threaded_simulator_equals_the_plain_one():
    # slabs of every chunk simulated on separate threads give the plain
    # simulator's bits, for ragged slab splits and both input types
    for dt, K, C, threads in (("bf16", 8, 1001, 5), ("f32", 4, 7, 3), ("f32", 3, 2, 4)):
        rng = np.random.default_rng(C)
        x = [rng.standard_normal(K * C).astype(np.float32) for _ in range(K)]
        if dt == "bf16":
            x = [workloads.to_bf16_bits(a) for a in x]
        a32, a16 = oracle.reduce_scatter(x, 1.0 / K)
        b32, b16 = oracle.reduce_scatter_threaded(x, 1.0 / K, threads=threads)
        for c in range(K):
            assert np.array_equal(a32[c].view(np.uint32), b32[c].view(np.uint32))
            assert np.array_equal(a16[c], b16[c])


# --------------------------------------------------------------------------
# Data-parallel weight gradient (fp64 reference)
# --------------------------------------------------------------------------

def pin_wgrad_brute_force_tiny():
    # dW[f, d] = sum over ranks and tokens of dy[t, f] * x[t, d], by plain loops
    K, T, F, D = 3, 5, 4, 6
    dys, xs = workloads.wgrad_operands(T, F, D, K)
    got = oracle.wgrad_psum_f64(dys, xs, scale=0.5)
    dyf = [oracle.bf16_widen(a).astype(np.float64).tolist() for a in dys]
    xf = [oracle.bf16_widen(a).astype(np.float64).tolist() for a in xs]
    for f in range(F):
        for d in range(D):
            acc = 0.0
            for r in range(K):
                for t in range(T):
                    acc += dyf[r][t][f] * xf[r][t][d]
            assert abs(got[f, d] - 0.5 * acc) <= 1e-12 * max(1.0, abs(acc))


def pin_wgrad_is_the_unsharded_gradient():
    # data parallelism splits the tokens: the gradient over all ranks' tokens
    # at once is dY^T X with the ranks' rows stacked (numpy fp64 matmul)
    dys, xs = workloads.wgrad_operands(T=10, F=24, D=16, K=4)
    got = oracle.wgrad_psum_f64(dys, xs)
    dy = np.concatenate([oracle.bf16_widen(a).astype(np.float64) for a in dys], axis=0)
    x = np.concatenate([oracle.bf16_widen(a).astype(np.float64) for a in xs], axis=0)
    assert np.allclose(got, dy.T @ x, rtol=1e-12, atol=1e-15)


def pin_wgrad_integer_exact_and_scaled():
    dys, xs = workloads.wgrad_operands(T=16, F=8, D=12, K=8, ints=True)
    got = oracle.wgrad_psum_f64(dys, xs, scale=0.125)
    dy = np.concatenate([oracle.bf16_widen(a).astype(np.int64) for a in dys], axis=0)
    x = np.concatenate([oracle.bf16_widen(a).astype(np.int64) for a in xs], axis=0)
    assert np.array_equal(got, (dy.T @ x).astype(np.float64) * 0.125)


# --------------------------------------------------------------------------
# Variable-length microbatch step
# --------------------------------------------------------------------------

def _odc_grads(K, N, m, seed):
    rng = np.random.default_rng(seed)
    return [[workloads.to_bf16_bits(rng.standard_normal(N).astype(np.float32) *
                                    np.float32(1e-3 * (j + 1))) for j in range(m[r])]
            for r in range(K)]


def pin_padding_buckets_are_neutral():
    K, N = 8, 8 * 64
    m = [1, 3, 2, 8, 5, 1, 7, 4]
    grads = _odc_grads(K, N, m, 11)
    M = max(m)
    padded = [g + [None] * (M - len(g)) for g in grads]
    a32, a16 = oracle.odc_layer(grads, m, 1.0 / K, N)
    b32, b16 = oracle.odc_layer(padded, [M] * K, 1.0 / K, N)
    for c in range(K):
        assert np.array_equal(_bits(a32[c]), _bits(b32[c]))
        assert np.array_equal(a16[c], b16[c])


def pin_one_microbatch_is_plain_reduce_scatter():
    K, N = 4, 4 * 32
    m = [1] * K
    grads = _odc_grads(K, N, m, 12)
    a32, _ = oracle.odc_layer(grads, m, 0.25, N)
    b32, _ = oracle.reduce_scatter([g[0] for g in grads], 0.25)
    for c in range(K):
        assert np.array_equal(_bits(a32[c]), _bits(b32[c]))


def pin_accumulator_integer_exact_and_plus_zero():
    rng = np.random.default_rng(13)
    gs = [rng.integers(-8, 9, 200).astype(np.float32) for _ in range(5)]
    acc = np.full(200, 123.0, np.float32)
    oracle.accumulate(acc, gs[0], first=True)
    for g in gs[1:]:
        oracle.accumulate(acc, g, first=False)
    assert np.array_equal(acc, np.sum(np.stack(gs), axis=0).astype(np.float32))
    # a -0 gradient into a fresh (+0-seeded) accumulator gives +0
    acc2 = np.full(4, 7.0, np.float32)
    oracle.accumulate(acc2, np.full(4, -0.0, np.float32), first=True)
    assert np.all(acc2.view(np.uint32) == 0)
    # a padding bucket leaves the accumulator's bits unchanged
    before = acc.copy()
    oracle.accumulate(acc, None, first=False)
    assert np.array_equal(acc.view(np.uint32), before.view(np.uint32))


def _odc_golden(name):
    rows = _golden_rows(name)
    K, N = map(int, rows[0].split())
    per_rank = [[float(v) for v in rows[1 + r].split()] for r in range(K)]
    return K, N, per_rank, rows[1 + K:]


def _odc_golden_grads(K, N, per_rank, dtype):
    if dtype == "bf16":
        return [[workloads.to_bf16_bits(np.full(N, v, np.float32)) for v in vals]
                for vals in per_rank]
    return [[np.full(N, v, np.float32) for v in vals] for vals in per_rank]


def pin_odc_association_by_hand():
    """A rank's microbatches accumulate in ascending order into a +0-seeded
    fp32 sum, then one ring settle ("Using ODC to Accelerate AMD SFT
    Training", "From Per-iteration to Per-minibatch Synchronization"); the
    golden's other lines are what a settle per microbatch, a flat fold, a
    descending or a pairwise microbatch order would give instead."""
    K, N, per_rank, rest = _odc_golden("odc_association_k2.txt")
    expect = [float(v) for v in rest[0].split()]
    wrong = [float(v) for v in rest[1].split()]
    m = [len(v) for v in per_rank]
    for dt, code in (("bf16", oracle.BF16), ("f32", oracle.F32)):
        grads = _odc_golden_grads(K, N, per_rank, dt)
        f32, b16 = oracle.odc_layer(grads, m, 1.0, N, grad_dtype=code)
        got = [float(x) for s in f32 for x in s]
        assert got == expect, (got, "wrong readings give", wrong)
        assert oracle.bf16_widen(np.concatenate(b16)).tolist() == expect


def pin_odc_pipeline_by_hand():
    """Cross-iteration settle pipeline ("Discussion: Settle Does Not Yet
    Overlap with Backward"): per-group settles added to the owner's +0-seeded
    accumulator in group order."""
    K, N, per_rank, rest = _odc_golden("odc_pipeline_k2.txt")
    m = [len(v) for v in per_rank]
    for dt, code in (("bf16", oracle.BF16), ("f32", oracle.F32)):
        grads = _odc_golden_grads(K, N, per_rank, dt)
        for line in rest[:-1]:
            bounds, exp = line.split(";")
            bounds = [int(v) for v in bounds.split()]
            exp = [float(v) for v in exp.split()]
            f32, _ = oracle.odc_pipelined(grads, m, bounds, 1.0, N, grad_dtype=code)
            got = [float(x) for s in f32 for x in s]
            assert got == exp, (bounds, got, exp)


def pin_odc_pipeline_one_group_is_the_single_settle():
    K, N = 8, 8 * 48
    m = [1, 3, 2, 8, 5, 1, 7, 4]
    grads = _odc_grads(K, N, m, 14)
    a32, a16 = oracle.odc_layer(grads, m, 1.0 / K, N)
    b32, b16 = oracle.odc_pipelined(grads, m, [0, max(m)], 1.0 / K, N)
    for c in range(K):
        assert np.array_equal(_bits(a32[c]), _bits(b32[c]))
        assert np.array_equal(a16[c], b16[c])


def pin_odc_pipeline_integer_exact_average_once():
    """Integer-valued gradients: every partial sum is exact, so any grouping
    gives the exact sum; the average (1/3 here, not a power of two) must be
    one fp32 rounding of that sum, applied once at the end."""
    rng = np.random.default_rng(15)
    K, N = 4, 4 * 64
    m = [3, 5, 1, 4]
    grads = [[rng.integers(-8, 9, N).astype(np.float32) for _ in range(m[r])] for r in range(K)]
    exact = np.zeros(N, np.int64)
    for r in range(K):
        for g in grads[r]:
            exact += g.astype(np.int64)
    want = exact.astype(np.float32) * np.float32(1.0 / 3.0)
    for bounds in ([0, 5], [0, 2, 5], [0, 1, 2, 3, 4, 5], [0, 0, 3, 5]):
        f32, _ = oracle.odc_pipelined(grads, m, bounds, 1.0 / 3.0, N, grad_dtype=oracle.F32)
        assert np.array_equal(_bits(np.concatenate(f32)), _bits(want)), bounds


def pin_odc_pipeline_padding_buckets_are_neutral():
    K, N = 4, 4 * 32
    m = [2, 5, 1, 3]
    grads = _odc_grads(K, N, m, 16)
    M = max(m)
    padded = [g + [None] * (M - len(g)) for g in grads]
    for bounds in ([0, 2, 5], [0, 1, 3, 5]):
        a32, a16 = oracle.odc_pipelined(grads, m, bounds, 0.25, N)
        b32, b16 = oracle.odc_pipelined(padded, [M] * K, bounds, 0.25, N)
        for c in range(K):
            assert np.array_equal(_bits(a32[c]), _bits(b32[c]))
            assert np.array_equal(a16[c], b16[c])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_skipped_ring_step_is_reported_not_hung():
    """Failure model: one rank skips one send of the reduce-scatter phase;
    the simulator reports the missing message (status 3) instead of waiting."""
    bufs = workloads.ring_ints(K=4, N=64, seed=3)
    for rank in range(4):
        for step in range(3):
            assert oracle.reduce_scatter_with_skipped_step(bufs, rank, step) == 3
    assert oracle.reduce_scatter_with_skipped_step(bufs, -1, -1) == 0
