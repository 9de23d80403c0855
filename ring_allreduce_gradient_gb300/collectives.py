"""Tensor-level helpers over the C ABI: allocate outputs with PyTorch on the
inputs' device and call the binding.  No arithmetic happens here.

Each rank of the K virtual ranks is one CUDA tensor; a call covers all K.
"""
from __future__ import annotations

import torch

from . import binding as B

_DT = {torch.float32: B.DP_FP32, torch.bfloat16: B.DP_BF16}
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def _code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _check_ranks(ts):
    if not ts:
        raise ValueError("need at least one rank")
    n, dt, dev = ts[0].numel(), ts[0].dtype, ts[0].device
    for t in ts:
        if t.numel() != n or t.dtype != dt or t.device != dev or not t.is_contiguous():
            raise ValueError("ranks need contiguous tensors of one size, dtype and device")
    return n, dt, dev


def reduce_scatter(bufs, scale: float, out_dtypes=("f32", "bf16"), stream=None):
    """Ring reduce-scatter of K rank tensors; returns (fp32 shards, bf16 shards)."""
    N, _, dev = _check_ranks(bufs)
    K = len(bufs)
    C = N // K
    o32 = [torch.empty(C, dtype=torch.float32, device=dev) for _ in range(K)] \
        if "f32" in out_dtypes else None
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=dev) for _ in range(K)] \
        if "bf16" in out_dtypes else None
    B.dp_reduce_scatter_dual(bufs, K, N, _code(bufs[0]), o32, o16, scale, stream)
    return o32, o16


def all_gather(shards, stream=None, copy_engines: bool = False):
    """Ring all-gather of K shards into K buffers of K*C elements; with
    ``copy_engines`` the copies run on the GPU's DMA engines instead of its
    SMs (the same bits)."""
    C, dt, dev = _check_ranks(shards)
    K = len(shards)
    out = [torch.empty(K * C, dtype=dt, device=dev) for _ in range(K)]
    fn = B.dp_all_gather_copy_engine if copy_engines else B.dp_all_gather
    fn(shards, K, C, _code(shards[0]), out, stream)
    return out


def all_reduce_(bufs, scale: float, stream=None):
    """In-place ring all-reduce of K rank tensors."""
    N, _, _ = _check_ranks(bufs)
    B.dp_ring_allreduce(bufs, len(bufs), N, _code(bufs[0]), scale, stream)
    return bufs


# Workspaces of the tensor-core calls (the chained split of a part-full last
# round), one per (device, stream): calls on one stream never overlap, so they
# can share one.  The sizes the library asks for are cached per device, call
# and shape, and forgotten when the CTA limits change through the binding (a
# size left stale by a limit changed elsewhere only costs the split: the
# library runs a launch unsplit, with the same bits, when the workspace is
# too small for it).
_GEMM_WS: dict = {}
_WS_BYTES: dict = {}


def _workspace(workspace, device, st, key, query):
    """The workspace to pass: "auto" (a cached one per device and stream, of
    the size ``query()`` asks for), None (none: the same bits, unsplit), or the
    caller's device tensor.  ``st`` is the resolved stream handle, ``key``
    names the call and its shape."""
    if not isinstance(workspace, str):
        return workspace
    k = (device.index, B.limits_epoch) + key
    nbytes = _WS_BYTES.get(k)
    if nbytes is None:
        with torch.cuda.device(device):
            nbytes = query()
        _WS_BYTES[k] = nbytes
    if nbytes == 0:
        return None
    wk = (device.index, st)
    ws = _GEMM_WS.get(wk)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _GEMM_WS[wk] = ws
    return ws


def allgather_matmul(x: torch.Tensor, w_shards, y_dtype=torch.bfloat16, stream=None,
                     workspace="auto"):
    """y = x . w^T with w the row concatenation of the shards (bf16 in)."""
    M, D = x.shape
    K = len(w_shards)
    F_shard = w_shards[0].shape[0]
    y = torch.empty(M, K * F_shard, dtype=y_dtype, device=x.device)
    st = B._stream(stream)
    ws = _workspace(workspace, x.device, st, ("ag", M, D, K, F_shard),
                    lambda: B.dp_allgather_matmul_workspace_size(M, D, K, F_shard))
    B.dp_allgather_matmul(x, M, D, w_shards, K, F_shard, y, _DT[y_dtype], st, workspace=ws)
    return y


def matmul_allreduce(x_shards, w_shards, scale=1.0, y_dtype=torch.bfloat16, stream=None,
                     workspace="auto"):
    """Tensor-parallel psum fused into the GEMM; returns K identical [M, F] tensors."""
    K = len(x_shards)
    M, Ds = x_shards[0].shape
    F = w_shards[0].shape[0]
    dev = x_shards[0].device
    ys = [torch.empty(M, F, dtype=y_dtype, device=dev) for _ in range(K)]
    st = B._stream(stream)
    ws = _workspace(workspace, dev, st, ("mm", K, M, Ds, F),
                    lambda: B.dp_matmul_workspace_size(K, M, Ds, F))
    B.dp_matmul_allreduce(x_shards, w_shards, K, M, Ds, F, ys, _DT[y_dtype], scale, st,
                          workspace=ws)
    return ys


def matmul_reduce_scatter(x_shards, w_shards, scale=1.0, y_dtype=torch.bfloat16, stream=None,
                          workspace="auto"):
    """Tensor-parallel psum fused into the GEMM; returns K row shards [M/K, F]."""
    K = len(x_shards)
    M, Ds = x_shards[0].shape
    F = w_shards[0].shape[0]
    dev = x_shards[0].device
    ys = [torch.empty(M // K, F, dtype=y_dtype, device=dev) for _ in range(K)]
    st = B._stream(stream)
    ws = _workspace(workspace, dev, st, ("mm", K, M, Ds, F),
                    lambda: B.dp_matmul_workspace_size(K, M, Ds, F))
    B.dp_matmul_reduce_scatter(x_shards, w_shards, K, M, Ds, F, ys, _DT[y_dtype], scale, st,
                               workspace=ws)
    return ys


def matmul_allreduce_xw(x_shards, w_shards, scale=1.0, y_dtype=torch.bfloat16, stream=None,
                        workspace="auto"):
    """As matmul_allreduce with each rank's weight [D_shard, F] (y = x . w)."""
    K = len(x_shards)
    M, Ds = x_shards[0].shape
    F = w_shards[0].shape[1]
    dev = x_shards[0].device
    ys = [torch.empty(M, F, dtype=y_dtype, device=dev) for _ in range(K)]
    st = B._stream(stream)
    ws = _workspace(workspace, dev, st, ("xw", K, M, Ds, F),
                    lambda: B.dp_matmul_xw_workspace_size(K, M, Ds, F))
    B.dp_matmul_allreduce_xw(x_shards, w_shards, K, M, Ds, F, ys, _DT[y_dtype], scale, st,
                             workspace=ws)
    return ys


def matmul_reduce_scatter_xw(x_shards, w_shards, scale=1.0, y_dtype=torch.bfloat16,
                             stream=None, workspace="auto"):
    """As matmul_reduce_scatter with each rank's weight [D_shard, F] (y = x . w)."""
    K = len(x_shards)
    M, Ds = x_shards[0].shape
    F = w_shards[0].shape[1]
    dev = x_shards[0].device
    ys = [torch.empty(M // K, F, dtype=y_dtype, device=dev) for _ in range(K)]
    st = B._stream(stream)
    ws = _workspace(workspace, dev, st, ("xw", K, M, Ds, F),
                    lambda: B.dp_matmul_xw_workspace_size(K, M, Ds, F))
    B.dp_matmul_reduce_scatter_xw(x_shards, w_shards, K, M, Ds, F, ys, _DT[y_dtype], scale,
                                  st, workspace=ws)
    return ys


def wgrad_reduce_scatter(dy, x, scale=None, dw_dtype=torch.bfloat16, stream=None,
                         workspace="auto"):
    """FSDP backward weight gradient fused with its reduce-scatter: rank r's
    dy[r] [T, F] and x[r] [T, D] (bf16); returns K row shards [F/K, D] of
    dW = scale * sum_r dy[r]^T x[r] (scale defaults to 1/K).  ``workspace``:
    "auto" (a cached one per device and stream, of the size the library asks
    for), None (no split of the last round; the same bits), or a device tensor."""
    K = len(dy)
    T, F = dy[0].shape
    D = x[0].shape[1]
    s = 1.0 / K if scale is None else scale
    dev = dy[0].device
    out = [torch.empty(F // K, D, dtype=dw_dtype, device=dev) for _ in range(K)]
    st = B._stream(stream)
    ws = _workspace(workspace, dev, st, ("wg", K, T, F, D),
                    lambda: B.dp_wgrad_workspace_size(K, T, F, D))
    B.dp_wgrad_reduce_scatter(dy, x, K, T, F, D, out, _DT[dw_dtype], s, st, workspace=ws)
    return out


def grad_accumulate_(acc: torch.Tensor, grad, first: bool, stream=None):
    code = _code(grad) if grad is not None else B.DP_BF16
    B.dp_grad_accumulate(acc, grad, acc.numel(), code, first, stream)
    return acc


def odc_reduce_scatter(grads, m, N: int, scale: float, grad_dtype=torch.bfloat16,
                       out_dtypes=("f32", "bf16"), device=None, stream=None):
    """Fused accumulate + settle.  ``grads[r]`` is rank r's list of microbatch
    gradients (tensors, or None for a padding bucket); rank r runs m[r]."""
    K = len(grads)
    Mmax = max([len(g) for g in grads] + [0])
    table = []
    for r in range(K):
        row = list(grads[r]) + [None] * (Mmax - len(grads[r]))
        table.extend(row)
    if device is None:
        device = next(t.device for t in table if t is not None)
    C = N // K
    o32 = [torch.empty(C, dtype=torch.float32, device=device) for _ in range(K)] \
        if "f32" in out_dtypes else None
    o16 = [torch.empty(C, dtype=torch.bfloat16, device=device) for _ in range(K)] \
        if "bf16" in out_dtypes else None
    B.dp_odc_reduce_scatter(table, m, K, Mmax, N, _DT[grad_dtype], o32, o16, scale, stream)
    return o32, o16


def _group_table(grads):
    """Row-major K x Mmax pointer table of one microbatch group."""
    K = len(grads)
    Mmax = max([len(g) for g in grads] + [0])
    table = []
    for r in range(K):
        table.extend(list(grads[r]) + [None] * (Mmax - len(grads[r])))
    return table, [len(g) for g in grads], Mmax


def odc_settle_group(grads, N: int, owner_acc, phase: int, scale: float, out=None,
                     grad_dtype=torch.bfloat16, stream=None):
    """One group of a pipelined settle on ``stream``: ``grads[r]`` is rank r's
    list of this group's microbatch gradients; ``owner_acc`` the K fp32
    owner accumulators; ``out`` the (f32, bf16) shard lists for a last
    group."""
    table, m, Mmax = _group_table(grads)
    K = len(grads)
    o32, o16 = out if out is not None else (None, None)
    B.dp_odc_settle_group(table, m, K, Mmax, N, _DT[grad_dtype], owner_acc, phase, o32, o16,
                          scale, stream)


class SettlePipe:
    """Cross-iteration settle pipeline over K virtual ranks ("Using ODC to
    Accelerate AMD SFT Training", "Discussion: Settle Does Not Yet Overlap
    with Backward"): each pushed microbatch group is settled on the library's
    side stream after the caller's stream reaches the push, while the caller
    goes on with the next group's backward; ``wait`` is the once-per-minibatch
    join.  The owner accumulators and the outputs are torch allocations made
    here; the library allocates no device memory."""

    def __init__(self, K: int, N: int, device, cta_limit: int = 0,
                 out_dtypes=("f32", "bf16")):
        _, self.handle = B.dp_settle_pipe_create(cta_limit)
        self.K, self.N = K, N
        C = N // K
        self.acc = [torch.empty(C, dtype=torch.float32, device=device) for _ in range(K)]
        self.out32 = [torch.empty(C, dtype=torch.float32, device=device) for _ in range(K)] \
            if "f32" in out_dtypes else None
        self.out16 = [torch.empty(C, dtype=torch.bfloat16, device=device) for _ in range(K)] \
            if "bf16" in out_dtypes else None

    def push(self, grads, first: bool, last: bool, scale: float, grad_dtype=torch.bfloat16,
             stream=None):
        """Settle one group (``grads[r]``: rank r's microbatches of the group);
        returns at once.  After the last group's push and a ``wait``, the
        outputs ``out32`` / ``out16`` hold the averaged shards."""
        table, m, Mmax = _group_table(grads)
        phase = (B.DP_SETTLE_FIRST if first else 0) | (B.DP_SETTLE_LAST if last else 0)
        B.dp_settle_pipe_push(self.handle, table, m, self.K, Mmax, self.N, _DT[grad_dtype],
                              self.acc, phase, self.out32, self.out16, scale, stream)

    def wait(self, stream=None):
        B.dp_settle_pipe_wait(self.handle, stream)

    def close(self):
        h = getattr(self, "handle", 0)
        if h:
            self.handle = 0
            B.dp_settle_pipe_destroy(h)

    def __del__(self):
        self.close()


def bucket_allreduce_(tensors_by_rank, scale: float, stream=None):
    """In-place all-reduce of one bucket; ``tensors_by_rank[r]`` is rank r's
    list of gradient tensors (the bucket's order)."""
    K = len(tensors_by_rank)
    n = len(tensors_by_rank[0])
    grads = [tensors_by_rank[r][t] for t in range(n) for r in range(K)]
    numels = [tensors_by_rank[0][t].numel() for t in range(n)]
    B.dp_bucket_allreduce(grads, numels, n, K, _code(tensors_by_rank[0][0]), scale, stream)
    return tensors_by_rank


class Reducer:
    """DDP-style gradient reducer over K virtual ranks (host logic in the C
    library: bucket assignment, pending counts, in-order launches)."""

    def __init__(self, numels, dtype, K: int, bucket_cap_bytes: int = 25 * 1024 * 1024,
                 scale: float = 1.0):
        _, self.handle = B.dp_reducer_create(list(numels), len(numels), _DT.get(dtype, dtype), K,
                                             bucket_cap_bytes, scale)
        self.K = K

    def __del__(self):
        h = getattr(self, "handle", 0)
        if h:
            B.dp_reducer_destroy(h)
            self.handle = 0

    @property
    def num_buckets(self) -> int:
        return B.dp_reducer_num_buckets(self.handle)

    def bucket_info(self, b):
        _, n, ne = B.dp_reducer_bucket_info(self.handle, b)
        return n, ne

    def param_slot(self, p):
        _, b, off = B.dp_reducer_param_slot(self.handle, p)
        return b, off

    def mark_ready(self, p, grads, stream=None) -> int:
        _, n = B.dp_reducer_mark_ready(self.handle, p, grads, stream)
        return n

    def finish(self):
        return B.dp_reducer_finish(self.handle)

    def set_dry_run(self, on: bool):
        B.dp_reducer_set_dry_run(self.handle, on)

    def set_overlap(self, on: bool):
        """Reduce buckets on the reducer's own streams (two, alternating)
        while the caller's stream goes on with the backward (DDP's
        asynchronous all-reduce)."""
        B.dp_reducer_set_overlap(self.handle, on)

    def wait(self, stream=None):
        """The join before the optimizer step: ``stream`` waits for every
        bucket launched so far."""
        B.dp_reducer_wait(self.handle, stream)

    def launch_log(self):
        return B.dp_reducer_launch_log(self.handle)
