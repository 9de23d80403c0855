"""Thin ctypes binding of the C ABI in ``include/dp.h``.

Each function has the C entry point's name and arguments and only marshals
them: Python sequences of device pointers become the host pointer arrays the
ABI takes, tensors are passed by ``data_ptr()``, and ``stream=None`` means
PyTorch's current CUDA stream.  All work happens in ``libdp_gb300.so``; there
is no other implementation behind these names, and loading fails loudly when
the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

DP_FP32 = 0
DP_BF16 = 1
DP_MAX_K = 16
DP_MAX_MICROBATCHES = 16
DP_WGRAD_NOALLOC_MAX_BYTES = 8 << 20  # the built-in scratch of the no-allocation call

DP_OK = 0
DP_ERR_INVALID_ARG = 1
DP_ERR_UNSUPPORTED = 2
DP_ERR_ALIAS = 3
DP_ERR_CUDA = 4
DP_ERR_TIMEOUT = 5

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdp_gb300.so")

_lock = threading.Lock()
_lib = None


class DpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libdp_gb300.so (built in-tree by ``build.py``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
        pp = ctypes.POINTER(ctypes.c_void_p)
        sig = {
            "dp_ring_allreduce": [pp, i32, sz, i32, f32, vp],
            "dp_reduce_scatter": [pp, i32, sz, i32, pp, f32, i32, vp],
            "dp_reduce_scatter_dual": [pp, i32, sz, i32, pp, pp, f32, vp],
            "dp_all_gather": [pp, i32, sz, i32, pp, vp],
            "dp_allgather_matmul": [vp, i32, i32, pp, i32, i32, vp, i32, vp, sz, vp],
            "dp_allgather_matmul_workspace_size": [i32, i32, i32, i32,
                                                   ctypes.POINTER(ctypes.c_size_t)],
            "dp_grad_accumulate": [vp, vp, sz, i32, i32, vp],
            "dp_matmul_allreduce": [pp, pp, i32, i32, i32, i32, pp, i32, f32, vp, sz, vp],
            "dp_matmul_reduce_scatter": [pp, pp, i32, i32, i32, i32, pp, i32, f32, vp, sz, vp],
            "dp_matmul_workspace_size": [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
            "dp_matmul_allreduce_xw": [pp, pp, i32, i32, i32, i32, pp, i32, f32, vp, sz, vp],
            "dp_matmul_reduce_scatter_xw": [pp, pp, i32, i32, i32, i32, pp, i32, f32, vp, sz,
                                            vp],
            "dp_matmul_xw_workspace_size": [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
            "dp_wgrad_reduce_scatter": [pp, pp, i32, i32, i32, i32, pp, i32, f32, vp, sz, vp],
            "dp_wgrad_workspace_size": [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
            "dp_wgrad_reduce_scatter_noalloc": [pp, pp, i32, i32, i32, i32, pp, i32, f32, vp],
            "dp_odc_reduce_scatter": [pp, ctypes.POINTER(ctypes.c_int), i32, i32, sz, i32, pp, pp,
                                      f32, vp],
            "dp_odc_settle_group": [pp, ctypes.POINTER(ctypes.c_int), i32, i32, sz, i32, pp, i32,
                                    pp, pp, f32, vp],
            "dp_settle_pipe_create": [i32, ctypes.POINTER(ctypes.c_void_p)],
            "dp_settle_pipe_push": [vp, pp, ctypes.POINTER(ctypes.c_int), i32, i32, sz, i32, pp,
                                    i32, pp, pp, f32, vp],
            "dp_settle_pipe_wait": [vp, vp],
            "dp_settle_pipe_destroy": [vp],
            "dp_bucket_allreduce": [pp, ctypes.POINTER(ctypes.c_size_t), i32, i32, i32, f32, vp],
            "dp_reducer_create": [ctypes.POINTER(ctypes.c_size_t), i32, i32, i32, sz, f32,
                                  ctypes.POINTER(ctypes.c_void_p)],
            "dp_reducer_num_buckets": [vp],
            "dp_reducer_bucket_info": [vp, i32, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_size_t)],
            "dp_reducer_param_slot": [vp, i32, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_size_t)],
            "dp_reducer_mark_ready": [vp, i32, pp, vp, ctypes.POINTER(ctypes.c_int)],
            "dp_reducer_finish": [vp, ctypes.POINTER(ctypes.c_int)],
            "dp_reducer_set_dry_run": [vp, i32],
            "dp_reducer_launch_log": [vp, ctypes.POINTER(ctypes.c_int), i32],
            "dp_reducer_set_overlap": [vp, i32],
            "dp_reducer_wait": [vp, vp],
            "dp_all_gather_copy_engine": [pp, i32, sz, i32, pp, vp],
            "dp_set_cta_limits": [i32, i32],
            "dp_set_collective_variant": [i32],
            "dp_get_collective_variant": [],
            "dp_get_cta_limits": [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)],
            "dp_get_device_error": [vp],
            "dp_selftest_bounded_wait": [ctypes.c_uint32, vp],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = i32
        lib.dp_reducer_destroy.argtypes = [vp]
        lib.dp_reducer_destroy.restype = None
        lib.dp_status_string.argtypes = [i32]
        lib.dp_status_string.restype = ctypes.c_char_p
        lib.dp_version.argtypes = []
        lib.dp_version.restype = i32
        _lib = lib
        return lib


# --- marshalling helpers ------------------------------------------------------

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _parray(items) -> ctypes.Array:
    vals = [_ptr(x) for x in items]
    return (ctypes.c_void_p * max(1, len(vals)))(*vals)


_raw_stream = None  # torch's current-stream query without building a Stream object


def _stream(stream) -> int | None:
    global _raw_stream
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None  # nothing can be launched; host-only validation paths
        if _raw_stream is None:
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
        if _raw_stream:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


_DTYPE_CODES: dict = {}  # dtype (string or torch dtype) -> code, filled as they are seen


def dtype_code(dt) -> int:
    """DP_FP32 / DP_BF16 from an int, a string ('f32', 'bf16') or a torch dtype."""
    if isinstance(dt, int):
        return dt
    c = _DTYPE_CODES.get(dt)
    if c is not None:
        return c
    s = str(dt)
    if s in ("f32", "fp32", "float32", "torch.float32"):
        c = DP_FP32
    elif s in ("bf16", "bfloat16", "torch.bfloat16"):
        c = DP_BF16
    else:
        return 99  # the library reports DP_ERR_UNSUPPORTED
    _DTYPE_CODES[dt] = c
    return c


def _ret(status: int, where: str, check: bool) -> int:
    if check and status != DP_OK:
        raise DpError(status, where)
    return status


def status_string(status: int) -> str:
    return load().dp_status_string(int(status)).decode()


# --- entry points ---------------------------------------------------------------

def dp_ring_allreduce(bufs, K, N, dtype, scale, stream=None, check=True) -> int:
    st = load().dp_ring_allreduce(_parray(bufs), K, N, dtype_code(dtype), scale, _stream(stream))
    return _ret(st, "dp_ring_allreduce", check)


def dp_reduce_scatter(bufs, K, N, in_dtype, out_shards, scale, out_dtype, stream=None,
                      check=True) -> int:
    st = load().dp_reduce_scatter(_parray(bufs), K, N, dtype_code(in_dtype), _parray(out_shards),
                                  scale, dtype_code(out_dtype), _stream(stream))
    return _ret(st, "dp_reduce_scatter", check)


def dp_reduce_scatter_dual(bufs, K, N, in_dtype, out_f32, out_bf16, scale, stream=None,
                           check=True) -> int:
    st = load().dp_reduce_scatter_dual(_parray(bufs), K, N, dtype_code(in_dtype),
                                       _parray(out_f32) if out_f32 is not None else None,
                                       _parray(out_bf16) if out_bf16 is not None else None,
                                       scale, _stream(stream))
    return _ret(st, "dp_reduce_scatter_dual", check)


def dp_all_gather(shards, K, shard_elems, dtype, out, stream=None, check=True) -> int:
    st = load().dp_all_gather(_parray(shards), K, shard_elems, dtype_code(dtype), _parray(out),
                              _stream(stream))
    return _ret(st, "dp_all_gather", check)


def _ws(workspace, workspace_bytes):
    """(pointer, bytes) of an optional workspace: a device tensor (bytes default
    to its size) or a raw pointer (bytes default to 0)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    return _ptr(workspace), workspace_bytes


def dp_allgather_matmul(x_local, M, D, w_shards, K, F_shard, y, y_dtype, stream=None,
                        check=True, workspace=None, workspace_bytes=None) -> int:
    wp, wb = _ws(workspace, workspace_bytes)
    st = load().dp_allgather_matmul(_ptr(x_local), M, D, _parray(w_shards), K, F_shard, _ptr(y),
                                    dtype_code(y_dtype), wp, wb, _stream(stream))
    return _ret(st, "dp_allgather_matmul", check)


def dp_matmul_allreduce(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale,
                        stream=None, check=True, workspace=None, workspace_bytes=None) -> int:
    wp, wb = _ws(workspace, workspace_bytes)
    st = load().dp_matmul_allreduce(_parray(x_shards), _parray(w_shards), K, M, D_shard, F,
                                    _parray(y_out), dtype_code(y_dtype), scale, wp, wb,
                                    _stream(stream))
    return _ret(st, "dp_matmul_allreduce", check)


def dp_matmul_reduce_scatter(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale,
                             stream=None, check=True, workspace=None,
                             workspace_bytes=None) -> int:
    wp, wb = _ws(workspace, workspace_bytes)
    st = load().dp_matmul_reduce_scatter(_parray(x_shards), _parray(w_shards), K, M, D_shard, F,
                                         _parray(y_out), dtype_code(y_dtype), scale, wp, wb,
                                         _stream(stream))
    return _ret(st, "dp_matmul_reduce_scatter", check)


def dp_matmul_allreduce_xw(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale,
                           stream=None, check=True, workspace=None, workspace_bytes=None) -> int:
    """The x . w orientation: ``w_shards[r]`` is [D_shard, F] row-major."""
    wp, wb = _ws(workspace, workspace_bytes)
    st = load().dp_matmul_allreduce_xw(_parray(x_shards), _parray(w_shards), K, M, D_shard, F,
                                       _parray(y_out), dtype_code(y_dtype), scale, wp, wb,
                                       _stream(stream))
    return _ret(st, "dp_matmul_allreduce_xw", check)


def dp_matmul_reduce_scatter_xw(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale,
                                stream=None, check=True, workspace=None,
                                workspace_bytes=None) -> int:
    wp, wb = _ws(workspace, workspace_bytes)
    st = load().dp_matmul_reduce_scatter_xw(_parray(x_shards), _parray(w_shards), K, M, D_shard,
                                            F, _parray(y_out), dtype_code(y_dtype), scale, wp, wb,
                                            _stream(stream))
    return _ret(st, "dp_matmul_reduce_scatter_xw", check)


def dp_matmul_xw_workspace_size(K, M, D_shard, F) -> int:
    n = ctypes.c_size_t(0)
    _ret(load().dp_matmul_xw_workspace_size(K, M, D_shard, F, ctypes.byref(n)),
         "dp_matmul_xw_workspace_size", True)
    return int(n.value)


def dp_allgather_matmul_workspace_size(M, D, K, F_shard) -> int:
    n = ctypes.c_size_t(0)
    _ret(load().dp_allgather_matmul_workspace_size(M, D, K, F_shard, ctypes.byref(n)),
         "dp_allgather_matmul_workspace_size", True)
    return int(n.value)


def dp_matmul_workspace_size(K, M, D_shard, F) -> int:
    n = ctypes.c_size_t(0)
    _ret(load().dp_matmul_workspace_size(K, M, D_shard, F, ctypes.byref(n)),
         "dp_matmul_workspace_size", True)
    return int(n.value)


def dp_wgrad_reduce_scatter(dy, x, K, T, F, D, dw_shards, dw_dtype, scale, stream=None,
                            check=True, workspace=None, workspace_bytes=None) -> int:
    """``workspace``: optional device tensor or pointer; ``workspace_bytes``
    defaults to the tensor's size (0 for a bare pointer)."""
    wp, wb = _ws(workspace, workspace_bytes)
    st = load().dp_wgrad_reduce_scatter(_parray(dy), _parray(x), K, T, F, D, _parray(dw_shards),
                                        dtype_code(dw_dtype), scale, wp, wb, _stream(stream))
    return _ret(st, "dp_wgrad_reduce_scatter", check)


def dp_wgrad_reduce_scatter_noalloc(dy, x, K, T, F, D, dw_shards, dw_dtype, scale, stream=None,
                                    check=True) -> int:
    """dp_wgrad_reduce_scatter for callers that cannot allocate device memory:
    its scratch is the library's built-in array (DP_WGRAD_NOALLOC_MAX_BYTES)."""
    st = load().dp_wgrad_reduce_scatter_noalloc(_parray(dy), _parray(x), K, T, F, D,
                                                _parray(dw_shards), dtype_code(dw_dtype), scale,
                                                _stream(stream))
    return _ret(st, "dp_wgrad_reduce_scatter_noalloc", check)


def dp_wgrad_workspace_size(K, T, F, D) -> int:
    n = ctypes.c_size_t(0)
    _ret(load().dp_wgrad_workspace_size(K, T, F, D, ctypes.byref(n)),
         "dp_wgrad_workspace_size", True)
    return int(n.value)


def dp_grad_accumulate(acc, grad, N, grad_dtype, first, stream=None, check=True) -> int:
    st = load().dp_grad_accumulate(_ptr(acc), _ptr(grad), N, dtype_code(grad_dtype),
                                   1 if first else 0, _stream(stream))
    return _ret(st, "dp_grad_accumulate", check)


def dp_odc_reduce_scatter(grads, m, K, Mmax, N, grad_dtype, out_f32, out_bf16, scale,
                          stream=None, check=True) -> int:
    """``grads``: flat row-major K*Mmax sequence of device pointers / tensors / None."""
    mm = (ctypes.c_int * max(1, K))(*[int(v) for v in m])
    st = load().dp_odc_reduce_scatter(_parray(grads), mm, K, Mmax, N, dtype_code(grad_dtype),
                                      _parray(out_f32) if out_f32 is not None else None,
                                      _parray(out_bf16) if out_bf16 is not None else None,
                                      scale, _stream(stream))
    return _ret(st, "dp_odc_reduce_scatter", check)


DP_SETTLE_FIRST = 1
DP_SETTLE_LAST = 2


def _opt_parray(a):
    return _parray(a) if a is not None else None


def dp_odc_settle_group(grads, m, K, Mmax, N, grad_dtype, owner_acc, phase, out_f32, out_bf16,
                        scale, stream=None, check=True) -> int:
    """One group of a pipelined settle; ``grads`` as for dp_odc_reduce_scatter
    (this group's microbatches only), ``owner_acc`` K fp32 shards or None."""
    mm = (ctypes.c_int * max(1, K))(*[int(v) for v in m])
    st = load().dp_odc_settle_group(_parray(grads), mm, K, Mmax, N, dtype_code(grad_dtype),
                                    _opt_parray(owner_acc), int(phase), _opt_parray(out_f32),
                                    _opt_parray(out_bf16), scale, _stream(stream))
    return _ret(st, "dp_odc_settle_group", check)


def dp_settle_pipe_create(cta_limit=0, check=True):
    """Returns (status, handle); handle is an opaque int (0 on failure)."""
    h = ctypes.c_void_p()
    st = load().dp_settle_pipe_create(int(cta_limit), ctypes.byref(h))
    _ret(st, "dp_settle_pipe_create", check)
    return st, (h.value or 0)


def dp_settle_pipe_push(h, grads, m, K, Mmax, N, grad_dtype, owner_acc, phase, out_f32, out_bf16,
                        scale, stream=None, check=True) -> int:
    mm = (ctypes.c_int * max(1, K))(*[int(v) for v in m])
    st = load().dp_settle_pipe_push(h, _parray(grads), mm, K, Mmax, N, dtype_code(grad_dtype),
                                    _opt_parray(owner_acc), int(phase), _opt_parray(out_f32),
                                    _opt_parray(out_bf16), scale, _stream(stream))
    return _ret(st, "dp_settle_pipe_push", check)


def dp_settle_pipe_wait(h, stream=None, check=True) -> int:
    return _ret(load().dp_settle_pipe_wait(h, _stream(stream)), "dp_settle_pipe_wait", check)


def dp_settle_pipe_destroy(h, check=True) -> int:
    return _ret(load().dp_settle_pipe_destroy(h), "dp_settle_pipe_destroy", check)


def dp_bucket_allreduce(grads, numels, n, K, dtype, scale, stream=None, check=True) -> int:
    """``grads``: flat tensor-major n*K sequence (grads[t*K + r])."""
    ne = (ctypes.c_size_t * max(1, n))(*[int(v) for v in numels])
    st = load().dp_bucket_allreduce(_parray(grads), ne, n, K, dtype_code(dtype), scale,
                                    _stream(stream))
    return _ret(st, "dp_bucket_allreduce", check)


def dp_reducer_create(numels, P, dtype, K, bucket_cap_bytes, scale, check=True):
    """Returns (status, handle); handle is an opaque int (0 on failure)."""
    ne = (ctypes.c_size_t * max(1, P))(*[int(v) for v in numels])
    h = ctypes.c_void_p()
    st = load().dp_reducer_create(ne, P, dtype_code(dtype), K, bucket_cap_bytes, scale,
                                  ctypes.byref(h))
    _ret(st, "dp_reducer_create", check)
    return st, (h.value or 0)


def dp_reducer_destroy(h) -> None:
    load().dp_reducer_destroy(h)


def dp_reducer_set_overlap(h, on, check=True) -> int:
    return _ret(load().dp_reducer_set_overlap(h, int(bool(on))), "dp_reducer_set_overlap", check)


def dp_reducer_wait(h, stream=None, check=True) -> int:
    return _ret(load().dp_reducer_wait(h, _stream(stream)), "dp_reducer_wait", check)


def dp_reducer_num_buckets(h) -> int:
    return load().dp_reducer_num_buckets(h)


def dp_reducer_bucket_info(h, b, check=True):
    n = ctypes.c_int()
    ne = ctypes.c_size_t()
    st = load().dp_reducer_bucket_info(h, b, ctypes.byref(n), ctypes.byref(ne))
    _ret(st, "dp_reducer_bucket_info", check)
    return st, n.value, ne.value


def dp_reducer_param_slot(h, p, check=True):
    b = ctypes.c_int()
    off = ctypes.c_size_t()
    st = load().dp_reducer_param_slot(h, p, ctypes.byref(b), ctypes.byref(off))
    _ret(st, "dp_reducer_param_slot", check)
    return st, b.value, off.value


def dp_reducer_mark_ready(h, p, grads, stream=None, check=True):
    """Returns (status, buckets launched by this call)."""
    n = ctypes.c_int()
    st = load().dp_reducer_mark_ready(h, p, _parray(grads), _stream(stream), ctypes.byref(n))
    _ret(st, "dp_reducer_mark_ready", check)
    return st, n.value


def dp_reducer_finish(h):
    """Returns (status, first pending bucket or -1)."""
    fp = ctypes.c_int()
    st = load().dp_reducer_finish(h, ctypes.byref(fp))
    return st, fp.value


def dp_reducer_set_dry_run(h, on, check=True) -> int:
    return _ret(load().dp_reducer_set_dry_run(h, 1 if on else 0), "dp_reducer_set_dry_run", check)


def dp_reducer_launch_log(h) -> list:
    lib = load()
    n = lib.dp_reducer_launch_log(h, None, 0)
    buf = (ctypes.c_int * max(1, n))()
    lib.dp_reducer_launch_log(h, buf, n)
    return list(buf[:n])


def dp_all_gather_copy_engine(shards, K, shard_elems, dtype, out, stream=None,
                              check=True) -> int:
    st = load().dp_all_gather_copy_engine(_parray(shards), K, shard_elems, dtype_code(dtype),
                                          _parray(out), _stream(stream))
    return _ret(st, "dp_all_gather_copy_engine", check)


# Bumped by every dp_set_cta_limits call made through this module: the
# workspace sizes a caller caches follow the GEMM CTA limit.
limits_epoch = 0


def dp_set_cta_limits(gemm_ctas, stream_ctas, check=True) -> int:
    global limits_epoch
    limits_epoch += 1
    return _ret(load().dp_set_cta_limits(int(gemm_ctas), int(stream_ctas)), "dp_set_cta_limits",
                check)


def dp_set_collective_variant(variant, check=True) -> int:
    return _ret(load().dp_set_collective_variant(int(variant)), "dp_set_collective_variant",
                check)


def dp_get_collective_variant() -> int:
    return load().dp_get_collective_variant()


def dp_get_cta_limits():
    g, s = ctypes.c_int(), ctypes.c_int()
    load().dp_get_cta_limits(ctypes.byref(g), ctypes.byref(s))
    return g.value, s.value


def dp_get_device_error(stream=None) -> int:
    return load().dp_get_device_error(_stream(stream))


def dp_selftest_bounded_wait(timeout_us, stream=None, check=True) -> int:
    st = load().dp_selftest_bounded_wait(int(timeout_us), _stream(stream))
    return _ret(st, "dp_selftest_bounded_wait", check)


def dp_version() -> int:
    return load().dp_version()
