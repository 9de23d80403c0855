"""CPU oracle for the ring reduce-scatter / all-gather / all-reduce path, the
FSDP all-gather + local GEMM and the variable-length microbatch step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and the product path never calls it.

The arithmetic lives in ``ring_oracle.c`` (plain scalar C, fp32 exactly as
written, fp64 for the GEMM reference); this module only builds that file with
gcc and marshals numpy arrays through ctypes.  bf16 values travel as their raw
16-bit patterns in ``numpy.uint16`` arrays.

Pages followed (cited per routine in ``ring_oracle.c``):
  * "CMU 11-868 L14-L15: Distributed Training and Data Parallelism, and Where
    Gradient Sync Costs Come From" -- "Ring AllReduce: ReduceScatter, then
    AllGather" (the step-by-step ring walk), "NCCL's five building blocks"
    (AllReduce = ReduceScatter + AllGather), "Intuition: data parallelism has
    only one thing to synchronize" (the average gradient).
  * "Sharding and Parallelism" -- "Real HLO before and after partitioning"
    (all-gather of w[64,512] shards, then the local dot).
  * "Using ODC to Accelerate AMD SFT Training" -- "From Per-iteration to
    Per-minibatch Synchronization" and "odc_pad vs odc_nopad" (Figure 5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c99", "-Wall", "-Wextra",
           "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None

# Mutation codes understood by oracle_set_mutation (tests only).
MUT_NONE = 0
MUT_REVERSED_RING = 1
MUT_START_AT_OWNER = 2
MUT_DROP_SCALE = 3
MUT_TRUNCATE_CAST = 4
MUT_SKIP_LAST_STEP = 5
MUT_GEMM_TRANSPOSE = 6
MUT_PAD_NOT_ZERO = 7
MUT_PSUM_SKIP_RANK = 8
MUT_ODC_SETTLE_PER_MB = 9
MUT_ODC_FLAT_FOLD = 10
MUT_ODC_REVERSED_MB = 11
MUT_ODC_PAIRWISE_MB = 12
MUT_PIPE_CARRY_IN_FOLD = 13
MUT_PIPE_REVERSED_GROUPS = 14
MUT_PIPE_SCALE_PER_GROUP = 15


def build(force: bool = False) -> str:
    """Compile ring_oracle.c into liboracle.so next to it (gcc, no GPU)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
        pp = ctypes.POINTER(ctypes.c_void_p)
        lib.oracle_set_mutation.argtypes = [i32]
        lib.oracle_set_mutation.restype = i32
        lib.oracle_bf16_round.argtypes = [f32]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_widen.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_widen.restype = f32
        for name in ("oracle_reduce_scatter_sim", "oracle_reduce_scatter_fold"):
            fn = getattr(lib, name)
            fn.argtypes = [pp, i32, sz, i32, f32, pp, pp]
            fn.restype = i32
        lib.oracle_reduce_scatter_sim_skip.argtypes = [pp, i32, sz, i32, f32, pp, pp, i32, i32]
        lib.oracle_reduce_scatter_sim_skip.restype = i32
        lib.oracle_all_gather_sim.argtypes = [pp, i32, sz, i32, pp]
        lib.oracle_all_gather_sim.restype = i32
        lib.oracle_all_reduce_sim.argtypes = [pp, i32, sz, i32, f32, pp]
        lib.oracle_all_reduce_sim.restype = i32
        lib.oracle_allgather_matmul_f64.argtypes = [vp, i32, i32, pp, i32, i32, vp]
        lib.oracle_allgather_matmul_f64.restype = i32
        lib.oracle_allgather_matmul_f64_sampled.argtypes = [vp, i32, i32, pp, i32, i32, vp, vp,
                                                            ctypes.c_int64, vp]
        lib.oracle_allgather_matmul_f64_sampled.restype = i32
        lib.oracle_matmul_psum_f64_sampled.argtypes = [pp, pp, i32, i32, i32, i32,
                                                       ctypes.c_double, vp, vp, ctypes.c_int64,
                                                       vp]
        lib.oracle_matmul_psum_f64_sampled.restype = i32
        lib.oracle_accumulate.argtypes = [vp, vp, sz, i32, i32]
        lib.oracle_accumulate.restype = i32
        lib.oracle_odc_layer.argtypes = [pp, ctypes.POINTER(ctypes.c_int), i32, i32, sz, i32, f32,
                                         pp, pp]
        lib.oracle_odc_layer.restype = i32
        ip = ctypes.POINTER(ctypes.c_int)
        lib.oracle_odc_pipelined.argtypes = [pp, ip, i32, i32, sz, i32, ip, i32, f32, pp, pp]
        lib.oracle_odc_pipelined.restype = i32
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


def _check(st: int, what: str) -> None:
    if st != 0:
        raise OracleError(f"{what} failed with status {st}")


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (raw bf16) arrays, got {a.dtype}")


def _ptrs(arrays) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(arrays))()
    for i, a in enumerate(arrays):
        arr[i] = a.ctypes.data if a is not None else None
    return arr


def _contig(arrays):
    return [np.ascontiguousarray(a) for a in arrays]


def set_mutation(m: int) -> int:
    """Plant a known mistake in the oracle (tests only); returns the old code."""
    return _load().oracle_set_mutation(int(m))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns (nearest, ties to even)."""
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = lib.oracle_bf16_round(float(v))
    return out.reshape(np.shape(x))


def bf16_widen(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns to float32 values (exact)."""
    lib = _load()
    flat = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(flat.shape, dtype=np.float32)
    for i, v in enumerate(flat):
        out[i] = lib.oracle_bf16_widen(int(v))
    return out.reshape(np.shape(h))


def _rs(name, bufs, scale, out_dtypes):
    lib = _load()
    bufs = _contig(bufs)
    K = len(bufs)
    N = bufs[0].size
    dt = _dtype_code(bufs[0])
    if any(b.size != N or b.dtype != bufs[0].dtype for b in bufs):
        raise ValueError("all ranks need the same size and dtype")
    if N % K:
        raise ValueError("reduce-scatter needs N % K == 0")
    C = N // K
    o32 = [np.empty(C, np.float32) for _ in range(K)] if "f32" in out_dtypes else None
    o16 = [np.empty(C, np.uint16) for _ in range(K)] if "bf16" in out_dtypes else None
    st = getattr(lib, name)(_ptrs(bufs), K, N, dt, float(scale),
                            _ptrs(o32) if o32 else None, _ptrs(o16) if o16 else None)
    _check(st, name)
    return o32, o16


def reduce_scatter(bufs, scale=1.0, out_dtypes=("f32", "bf16")):
    """Ring reduce-scatter by step simulation.

    ``bufs``: K equal-size 1-D arrays (float32, or uint16 raw bf16).
    Returns ``(shards_f32, shards_bf16)``: lists of K arrays of N/K elements
    (either is None when not requested).  Shard c = the chunk rank c holds
    after K-1 ring steps, times ``scale``, rounded to the output type.
    """
    return _rs("oracle_reduce_scatter_sim", bufs, scale, out_dtypes)


def reduce_scatter_threaded(bufs, scale=1.0, out_dtypes=("f32", "bf16"), threads=None):
    """The same step simulation on ``threads`` slabs at once.

    Every element's result depends only on its chunk and the K values at its
    offset, so the simulator is run unchanged on slabs: slab j takes the same
    element range [a_j, b_j) of every chunk of every rank, forming K buffers
    of K*(b_j - a_j) elements whose chunk c is chunk c's range.  The calls
    release the GIL, so they run on separate cores; the slab results are put
    back in place (no arithmetic outside the simulator)."""
    bufs = _contig(bufs)
    K, N = len(bufs), bufs[0].size
    if N % K:
        raise ValueError("reduce-scatter needs N % K == 0")
    C = N // K
    threads = max(1, min(threads or len(os.sched_getaffinity(0)), C))
    edges = [C * j // threads for j in range(threads + 1)]
    o32 = [np.empty(C, np.float32) for _ in range(K)] if "f32" in out_dtypes else None
    o16 = [np.empty(C, np.uint16) for _ in range(K)] if "bf16" in out_dtypes else None

    def run(j):
        a, b = edges[j], edges[j + 1]
        if a == b:
            return
        sub = [np.ascontiguousarray(x.reshape(K, C)[:, a:b]).reshape(-1) for x in bufs]
        s32, s16 = reduce_scatter(sub, scale, out_dtypes)
        for c in range(K):
            if o32 is not None:
                o32[c][a:b] = s32[c]
            if o16 is not None:
                o16[c][a:b] = s16[c]

    pool = [threading.Thread(target=run, args=(j,)) for j in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    return o32, o16


def reduce_scatter_with_skipped_step(bufs, skip_rank, skip_step, scale=1.0):
    """The ring walk with rank ``skip_rank`` skipping step ``skip_step``:
    returns the status (3 = a message never arrived) instead of hanging."""
    lib = _load()
    bufs = _contig(bufs)
    K, N = len(bufs), bufs[0].size
    C = N // K
    o32 = [np.empty(C, np.float32) for _ in range(K)]
    return lib.oracle_reduce_scatter_sim_skip(_ptrs(bufs), K, N, _dtype_code(bufs[0]),
                                              float(scale), _ptrs(o32), None, int(skip_rank),
                                              int(skip_step))


def reduce_scatter_fold(bufs, scale=1.0, out_dtypes=("f32", "bf16")):
    """The same result from the closed-form per-element fold."""
    return _rs("oracle_reduce_scatter_fold", bufs, scale, out_dtypes)


def all_gather(shards):
    """Ring all-gather by step simulation: K shards of C elements -> K
    buffers, each the concatenation shard_0 .. shard_{K-1}."""
    lib = _load()
    shards = _contig(shards)
    K = len(shards)
    C = shards[0].size
    dt = _dtype_code(shards[0])
    out = [np.zeros(K * C, shards[0].dtype) for _ in range(K)]
    _check(lib.oracle_all_gather_sim(_ptrs(shards), K, C, dt, _ptrs(out)), "all_gather")
    return out


def all_reduce(bufs, scale=1.0):
    """Ring all-reduce by step simulation (reduce-scatter, average and cast,
    all-gather).  Any N; returns K new arrays of the input dtype."""
    lib = _load()
    bufs = _contig(bufs)
    K = len(bufs)
    N = bufs[0].size
    dt = _dtype_code(bufs[0])
    out = [np.zeros(N, bufs[0].dtype) for _ in range(K)]
    _check(lib.oracle_all_reduce_sim(_ptrs(bufs), K, N, dt, float(scale), _ptrs(out)),
           "all_reduce")
    return out


def bucket_all_reduce(tensors_by_rank, scale=1.0):
    """Ring all-reduce of a DDP bucket: rank r's tensors concatenated in order
    form one flat buffer, which is all-reduced as a whole; returns the
    per-rank lists of tensors cut back out of the result."""
    K = len(tensors_by_rank)
    sizes = [np.asarray(t).size for t in tensors_by_rank[0]]
    flat = [np.concatenate([np.ascontiguousarray(t).ravel() for t in tensors_by_rank[r]])
            for r in range(K)]
    out = all_reduce(flat, scale)
    cuts = np.cumsum([0] + sizes)
    return [[out[r][cuts[i]:cuts[i + 1]] for i in range(len(sizes))] for r in range(K)]


def allgather_matmul_f64(x: np.ndarray, w_shards) -> np.ndarray:
    """FSDP forward: gather the K row shards w_k[F_shard, D] (uint16 raw bf16)
    and return y = x . w^T in float64, shape [M, K*F_shard]."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w_shards = [np.ascontiguousarray(w, dtype=np.uint16) for w in w_shards]
    M, D = x.shape
    K = len(w_shards)
    F_shard = w_shards[0].shape[0]
    y = np.empty((M, K * F_shard), np.float64)
    _check(lib.oracle_allgather_matmul_f64(x.ctypes.data, M, D, _ptrs(w_shards), K, F_shard,
                                           y.ctypes.data), "allgather_matmul_f64")
    return y


def allgather_matmul_f64_sampled(x, w_shards, ms, fs) -> np.ndarray:
    """y[ms[t], fs[t]] of the FSDP forward product, in float64."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w_shards = [np.ascontiguousarray(w, dtype=np.uint16) for w in w_shards]
    M, D = x.shape
    K = len(w_shards)
    F_shard = w_shards[0].shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    fs = np.ascontiguousarray(fs, dtype=np.int64)
    out = np.empty(ms.size, np.float64)
    _check(lib.oracle_allgather_matmul_f64_sampled(x.ctypes.data, M, D, _ptrs(w_shards), K,
                                                   F_shard, ms.ctypes.data, fs.ctypes.data,
                                                   ms.size, out.ctypes.data),
           "allgather_matmul_f64_sampled")
    return out


def matmul_psum_f64_sampled(x_shards, w_shards, ms, fs, scale=1.0) -> np.ndarray:
    """Tensor-parallel psum: y[ms[t], fs[t]] = scale * sum_r x_r . w_r^T, fp64.
    x_shards[r] [M, Ds] and w_shards[r] [F, Ds] are uint16 (raw bf16)."""
    lib = _load()
    xs = [np.ascontiguousarray(x, dtype=np.uint16) for x in x_shards]
    ws = [np.ascontiguousarray(w, dtype=np.uint16) for w in w_shards]
    K = len(xs)
    M, Ds = xs[0].shape
    F = ws[0].shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    fs = np.ascontiguousarray(fs, dtype=np.int64)
    out = np.empty(ms.size, np.float64)
    _check(lib.oracle_matmul_psum_f64_sampled(_ptrs(xs), _ptrs(ws), K, M, Ds, F, float(scale),
                                              ms.ctypes.data, fs.ctypes.data, ms.size,
                                              out.ctypes.data), "matmul_psum_f64_sampled")
    return out


def matmul_psum_f64(x_shards, w_shards, scale=1.0) -> np.ndarray:
    """The whole [M, F] tensor-parallel psum in fp64."""
    M = np.asarray(x_shards[0]).shape[0]
    F = np.asarray(w_shards[0]).shape[0]
    mm, ff = np.meshgrid(np.arange(M), np.arange(F), indexing="ij")
    return matmul_psum_f64_sampled(x_shards, w_shards, mm.ravel(), ff.ravel(), scale).reshape(M, F)


def wgrad_psum_f64_sampled(dy, x, fs, ds, scale=1.0) -> np.ndarray:
    """The data-parallel weight gradient of a linear layer ("Using ODC to
    Accelerate AMD SFT Training", section "Why FSDP is Slow": each rank's full
    layer gradient, then its reduce-scatter), in fp64:
    dW[fs[t], ds[t]] = scale * sum_r sum_tok dy_r[tok, f] * x_r[tok, d].
    dy[r] [T, F] and x[r] [T, D] are uint16 (raw bf16).  It is the psum above
    with both operands transposed: sum_r (dy_r^T) . (x_r^T)^T."""
    dyt = [np.ascontiguousarray(np.asarray(a, dtype=np.uint16).T) for a in dy]
    xt = [np.ascontiguousarray(np.asarray(a, dtype=np.uint16).T) for a in x]
    return matmul_psum_f64_sampled(dyt, xt, fs, ds, scale)


def wgrad_psum_f64(dy, x, scale=1.0) -> np.ndarray:
    """The whole [F, D] weight gradient in fp64."""
    F = np.asarray(dy[0]).shape[1]
    D = np.asarray(x[0]).shape[1]
    ff, dd = np.meshgrid(np.arange(F), np.arange(D), indexing="ij")
    return wgrad_psum_f64_sampled(dy, x, ff.ravel(), dd.ravel(), scale).reshape(F, D)


def accumulate(acc: np.ndarray, grad, first: bool) -> np.ndarray:
    """One microbatch into an fp32 accumulator (in place, also returned).
    ``grad`` None is a padding bucket (+0)."""
    lib = _load()
    assert acc.dtype == np.float32 and acc.flags.c_contiguous
    if grad is not None:
        grad = np.ascontiguousarray(grad)
        dt = _dtype_code(grad)
        gp = grad.ctypes.data
    else:
        dt, gp = BF16, None
    _check(lib.oracle_accumulate(acc.ctypes.data, gp, acc.size, dt, int(bool(first))),
           "accumulate")
    return acc


def _grad_table(grads, N):
    """K x Mmax table of microbatch gradient pointers (None: padding)."""
    K = len(grads)
    Mmax = max([len(g) for g in grads] + [0])
    keep = []
    table = (ctypes.c_void_p * max(1, K * Mmax))()
    for r in range(K):
        for j, g in enumerate(grads[r]):
            if g is not None:
                g = np.ascontiguousarray(g)
                if g.size != N:
                    raise ValueError("gradient size mismatch")
                keep.append(g)
                table[r * Mmax + j] = g.ctypes.data
    return table, Mmax, keep


def _shard_outputs(K, N, out_dtypes):
    C = N // K
    o32 = [np.empty(C, np.float32) for _ in range(K)] if "f32" in out_dtypes else None
    o16 = [np.empty(C, np.uint16) for _ in range(K)] if "bf16" in out_dtypes else None
    return o32, o16


def odc_layer(grads, m, scale, N, grad_dtype=BF16, out_dtypes=("f32", "bf16")):
    """One layer of the variable-length step.

    ``grads``: list over ranks of lists of microbatch gradients (arrays, or
    None for a padding bucket); rank r runs the first ``m[r]`` entries of its
    list into a +0-seeded fp32 accumulator, then one ring reduce-scatter over
    the K accumulators with ``scale``.  Returns (shards_f32, shards_bf16).
    """
    lib = _load()
    K = len(grads)
    table, Mmax, _keep = _grad_table(grads, N)
    mm = (ctypes.c_int * K)(*[int(v) for v in m])
    o32, o16 = _shard_outputs(K, N, out_dtypes)
    _check(lib.oracle_odc_layer(table, mm, K, Mmax, N, grad_dtype, float(scale),
                                _ptrs(o32) if o32 else None, _ptrs(o16) if o16 else None),
           "odc_layer")
    return o32, o16


def odc_pipelined(grads, m, bounds, scale, N, grad_dtype=BF16, out_dtypes=("f32", "bf16")):
    """One layer of the variable-length step with the cross-iteration settle
    pipeline: microbatch groups [bounds[g], bounds[g+1]) of j, each settled
    (per-rank +0-seeded sums, then the ring reduce-scatter) and added to the
    owners' +0-seeded fp32 accumulators in group order; the average ``scale``
    and the casts once at the end.  Returns (shards_f32, shards_bf16)."""
    lib = _load()
    K = len(grads)
    table, Mmax, _keep = _grad_table(grads, N)
    mm = (ctypes.c_int * K)(*[int(v) for v in m])
    G = len(bounds) - 1
    bb = (ctypes.c_int * len(bounds))(*[int(v) for v in bounds])
    o32, o16 = _shard_outputs(K, N, out_dtypes)
    _check(lib.oracle_odc_pipelined(table, mm, K, Mmax, N, grad_dtype, bb, G, float(scale),
                                    _ptrs(o32) if o32 else None, _ptrs(o16) if o16 else None),
           "odc_pipelined")
    return o32, o16
