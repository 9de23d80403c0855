"""The C-ABI library builds, loads and exports every entry point include/dp.h
declares; invalid arguments are rejected on the host before any CUDA call.
No test here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

from ring_allreduce_gradient_gb300 import binding as B
from ring_allreduce_gradient_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dp.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\bDP_API\s+[\w\s\*]+?\b(dp_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("dp_ring_allreduce", "dp_reduce_scatter", "dp_all_gather", "dp_allgather_matmul",
              "dp_reduce_scatter_dual", "dp_grad_accumulate", "dp_odc_reduce_scatter",
              "dp_get_device_error", "dp_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(dp_\w+)$", out, flags=re.M))
    assert set(declared_functions()) == exported
    for n in declared_functions():
        assert hasattr(lib, n)


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "dp.h"\nint main(void){ return DP_OK + DP_MAX_K * 0; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-c", str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_status_strings(lib):
    for code, name in [(0, "DP_OK"), (1, "DP_ERR_INVALID_ARG"), (2, "DP_ERR_UNSUPPORTED"),
                       (3, "DP_ERR_ALIAS"), (4, "DP_ERR_CUDA"), (5, "DP_ERR_TIMEOUT")]:
        assert B.status_string(code) == name
    assert B.dp_version() >= 100


# Fake, never-dereferenced device addresses: validation must reject these
# calls before touching CUDA.
BASE = 0x7F0000000000
MiB = 1 << 20


def fake(i, off=0):
    return BASE + i * 64 * MiB + off


def test_reduce_scatter_validation(lib):
    bufs = [fake(r) for r in range(4)]
    outs = [fake(8 + r) for r in range(4)]
    kw = dict(stream=0, check=False)
    assert B.dp_reduce_scatter(bufs, 0, 16, B.DP_FP32, outs, 1.0, B.DP_FP32, **kw) == 1
    assert B.dp_reduce_scatter(bufs, 17, 16, B.DP_FP32, outs, 1.0, B.DP_FP32, **kw) == 1
    assert B.dp_reduce_scatter(bufs, 4, 18, B.DP_FP32, outs, 1.0, B.DP_FP32, **kw) == 1
    assert B.dp_reduce_scatter(bufs, 4, 16, 7, outs, 1.0, B.DP_FP32, **kw) == 2
    assert B.dp_reduce_scatter(bufs, 4, 16, B.DP_FP32, outs, 1.0, 7, **kw) == 2
    assert B.dp_reduce_scatter(bufs[:3] + [None], 4, 16, B.DP_FP32, outs, 1.0, B.DP_FP32,
                               **kw) == 1
    # an output shard inside rank 2's input buffer
    bad = outs[:3] + [fake(2, 8)]
    assert B.dp_reduce_scatter(bufs, 4, 1024, B.DP_FP32, bad, 1.0, B.DP_FP32, **kw) == 3
    # two output shards overlapping each other
    bad = [fake(8), fake(8, 16), fake(10), fake(11)]
    assert B.dp_reduce_scatter(bufs, 4, 1024, B.DP_FP32, bad, 1.0, B.DP_FP32, **kw) == 3
    # N == 0 is a no-op
    assert B.dp_reduce_scatter(bufs, 4, 0, B.DP_FP32, outs, 1.0, B.DP_FP32, **kw) == 0
    assert B.dp_reduce_scatter_dual(bufs, 4, 16, B.DP_FP32, None, None, 1.0, **kw) == 1


def test_all_gather_and_allreduce_validation(lib):
    kw = dict(stream=0, check=False)
    shards = [fake(r) for r in range(4)]
    outs = [fake(8 + r) for r in range(4)]
    assert B.dp_all_gather(shards, 4, 0, B.DP_FP32, outs, **kw) == 0
    assert B.dp_all_gather(shards, 4, 16, 9, outs, **kw) == 2
    assert B.dp_all_gather(shards, 4, 16, B.DP_FP32, [fake(8), fake(8, 4), fake(10), fake(11)],
                           **kw) == 3
    assert B.dp_all_gather(shards, 4, 16, B.DP_FP32, outs[:3] + [fake(1, 0)], **kw) == 3
    # all-reduce buffers must be pairwise disjoint
    assert B.dp_ring_allreduce([fake(0), fake(0, 4), fake(2), fake(3)], 4, 100, B.DP_FP32, 1.0,
                               **kw) == 3
    assert B.dp_ring_allreduce(shards, 4, 0, B.DP_FP32, 1.0, **kw) == 0
    assert B.dp_ring_allreduce(shards, 0, 10, B.DP_FP32, 1.0, **kw) == 1


def test_bucket_null_pointers_only_for_empty_tensors(lib):
    numels = (ctypes.c_size_t * 2)(0, 0)
    ptrs = (ctypes.c_void_p * 4)(None, None, None, None)
    # every tensor empty: nothing to do, NULL pointers accepted, no launch
    assert lib.dp_bucket_allreduce(ptrs, numels, 2, 2, B.DP_FP32, ctypes.c_float(0.5), None) == 0
    numels2 = (ctypes.c_size_t * 2)(0, 16)
    # a non-empty tensor with a NULL pointer is rejected before any launch
    assert lib.dp_bucket_allreduce(ptrs, numels2, 2, 2, B.DP_FP32, ctypes.c_float(0.5), None) == 1


def test_matmul_accumulate_odc_validation(lib):
    kw = dict(stream=0, check=False)
    ws = [fake(1 + k) for k in range(8)]
    assert B.dp_allgather_matmul(fake(0), 128, 500, ws, 8, 64, fake(20), B.DP_BF16, **kw) == 2
    assert B.dp_allgather_matmul(fake(0), 128, 512, ws, 8, 60, fake(20), B.DP_BF16, **kw) == 2
    assert B.dp_allgather_matmul(fake(0, 2), 128, 512, ws, 8, 64, fake(20), B.DP_BF16, **kw) == 2
    assert B.dp_allgather_matmul(fake(0), 128, 512, ws, 8, 64, fake(3, 64), B.DP_BF16, **kw) == 3
    assert B.dp_allgather_matmul(fake(0), 0, 512, ws, 8, 64, fake(20), B.DP_BF16, **kw) == 0
    # optional workspace: 16-byte aligned, overlapping no operand or output
    assert B.dp_allgather_matmul(fake(0), 128, 512, ws, 8, 64, fake(20), B.DP_BF16,
                                 workspace=fake(30, 8), workspace_bytes=4096, **kw) == 2
    assert B.dp_allgather_matmul(fake(0), 128, 512, ws, 8, 64, fake(20), B.DP_BF16,
                                 workspace=fake(20, 64), workspace_bytes=4096, **kw) == 3
    assert B.dp_allgather_matmul(fake(0), 128, 512, ws, 8, 64, fake(20), B.DP_BF16,
                                 workspace=fake(0, 256), workspace_bytes=4096, **kw) == 3
    assert B.dp_grad_accumulate(fake(0), fake(0, 4), 100, B.DP_BF16, 1, **kw) == 3
    assert B.dp_grad_accumulate(None, fake(1), 100, B.DP_BF16, 1, **kw) == 1
    table = [fake(r * 2 + j) for r in range(4) for j in range(2)]
    outs = [fake(30 + r) for r in range(4)]
    assert B.dp_odc_reduce_scatter(table, [1, 2, 3, 1], 4, 2, 64, B.DP_BF16, outs, None, 0.25,
                                   **kw) == 1  # m[2] > Mmax
    assert B.dp_odc_reduce_scatter(table, [1, 2, 2, 1], 4, 2, 66, B.DP_BF16, outs, None, 0.25,
                                   **kw) == 1  # N % K
    bad_out = outs[:3] + [fake(5, 16)]
    assert B.dp_odc_reduce_scatter(table, [1, 2, 2, 1], 4, 2, 64, B.DP_BF16, bad_out, None,
                                   0.25, **kw) == 3
    assert B.dp_selftest_bounded_wait(0, **kw) == 1
    xs = [fake(r) for r in range(4)]
    ws_ = [fake(4 + r) for r in range(4)]
    ys = [fake(8 + r) for r in range(4)]
    assert B.dp_matmul_allreduce(xs, ws_, 4, 128, 60, 64, ys, B.DP_BF16, 1.0, **kw) == 2
    assert B.dp_matmul_allreduce(xs, ws_, 4, 128, 64, 40, ys, B.DP_BF16, 1.0, **kw) == 2
    assert B.dp_matmul_reduce_scatter(xs, ws_, 4, 130, 64, 64, ys, B.DP_BF16, 1.0, **kw) == 1
    assert B.dp_matmul_allreduce(xs, ws_, 4, 128, 64, 64, ys[:3] + [fake(2, 16)], B.DP_BF16,
                                 1.0, **kw) == 3
    assert B.dp_matmul_allreduce(xs, ws_, 4, 0, 64, 64, ys, B.DP_BF16, 1.0, **kw) == 0
    assert B.dp_matmul_allreduce(xs, ws_, 4, 128, 64, 64, ys, B.DP_BF16, 1.0,
                                 workspace=fake(30, 4), workspace_bytes=4096, **kw) == 2
    assert B.dp_matmul_reduce_scatter(xs, ws_, 4, 128, 64, 64, ys, B.DP_BF16, 1.0,
                                      workspace=fake(9, 32), workspace_bytes=4096, **kw) == 3
    assert B.dp_matmul_reduce_scatter(xs, ws_, 4, 128, 64, 64, ys, B.DP_BF16, 1.0,
                                      workspace=fake(5, 32), workspace_bytes=4096, **kw) == 3
    # weight gradient + reduce-scatter: only paths that return before any device call
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 128, 60, ys, B.DP_BF16, 0.25, **kw) == 2
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 96, 64, ys, B.DP_BF16, 0.25, **kw) == 2
    assert B.dp_wgrad_reduce_scatter(xs[:3], ws_[:3], 3, 128, 128, 64, ys[:3], B.DP_BF16,
                                     1.0, **kw) == 1  # F % K
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, -1, 128, 64, ys, B.DP_BF16, 0.25, **kw) == 1
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 128, 64, ys, B.DP_FP32 + 7, 0.25,
                                     **kw) == 2
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 128, 64, ys[:3] + [fake(2, 16)],
                                     B.DP_BF16, 0.25, **kw) == 3
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 0, 64, ys, B.DP_BF16, 0.25, **kw) == 0
    # the optional workspace: 16-byte aligned, overlapping no operand or output
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 128, 64, ys, B.DP_BF16, 0.25,
                                     workspace=fake(20, 8), workspace_bytes=4096, **kw) == 2
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 128, 64, ys, B.DP_BF16, 0.25,
                                     workspace=fake(0, 64), workspace_bytes=4096, **kw) == 3
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 128, 64, ys, B.DP_BF16, 0.25,
                                     workspace=fake(9, 64), workspace_bytes=4096, **kw) == 3
    assert B.dp_wgrad_reduce_scatter(xs, ws_, 4, 128, 0, 64, ys, B.DP_BF16, 0.25,
                                     workspace=fake(20), workspace_bytes=4096, **kw) == 0


def test_wgrad_workspace_size_validation(lib):
    import ctypes
    n = ctypes.c_size_t(7)
    assert lib.dp_wgrad_workspace_size(4, 128, 128, 64, None) == B.DP_ERR_INVALID_ARG
    assert lib.dp_wgrad_workspace_size(0, 128, 128, 64, ctypes.byref(n)) == B.DP_ERR_INVALID_ARG
    assert n.value == 0
    assert lib.dp_wgrad_workspace_size(4, -1, 128, 64, ctypes.byref(n)) == B.DP_ERR_INVALID_ARG


def test_gemm_workspace_size_validation(lib):
    import ctypes
    n = ctypes.c_size_t(7)
    assert lib.dp_allgather_matmul_workspace_size(128, 512, 8, 64, None) == B.DP_ERR_INVALID_ARG
    assert lib.dp_allgather_matmul_workspace_size(128, 512, 0, 64,
                                                  ctypes.byref(n)) == B.DP_ERR_INVALID_ARG
    assert n.value == 0
    assert lib.dp_matmul_workspace_size(8, 128, 64, 64, None) == B.DP_ERR_INVALID_ARG
    assert lib.dp_matmul_workspace_size(17, 128, 64, 64, ctypes.byref(n)) == B.DP_ERR_INVALID_ARG
    assert lib.dp_matmul_workspace_size(8, -1, 64, 64, ctypes.byref(n)) == B.DP_ERR_INVALID_ARG


def test_settle_group_and_pipe_validation(lib):
    """The pipelined settle's checks run on the host before any device call:
    phase bits, the owner accumulators a phase needs, outputs for the last
    group, aliasing with the gradients and the outputs, N % K."""
    kw = dict(stream=0, check=False)
    K = 4
    table = [fake(r * 2 + j) for r in range(K) for j in range(2)]
    acc = [fake(20 + r) for r in range(K)]
    outs = [fake(30 + r) for r in range(K)]
    m = [1, 2, 0, 2]
    F, L = B.DP_SETTLE_FIRST, B.DP_SETTLE_LAST
    g = B.dp_odc_settle_group
    assert g(table, m, K, 2, 64, B.DP_BF16, acc, 4, None, None, 1.0, **kw) == 1  # phase bits
    assert g(table, m, K, 2, 64, B.DP_BF16, None, F, None, None, 1.0, **kw) == 1  # no acc
    assert g(table, m, K, 2, 64, B.DP_BF16, None, 0, None, None, 1.0, **kw) == 1
    assert g(table, m, K, 2, 64, B.DP_BF16, acc, L, None, None, 1.0, **kw) == 1  # no outputs
    assert g(table, m, K, 2, 64, B.DP_BF16, acc[:3] + [None], 0, None, None, 1.0, **kw) == 1
    assert g(table, m, K, 2, 66, B.DP_BF16, acc, 0, None, None, 1.0, **kw) == 1  # N % K
    assert g(table, [1, 3, 0, 2], K, 2, 64, B.DP_BF16, acc, 0, None, None, 1.0, **kw) == 1
    assert g(table, m, K, 2, 64, B.DP_BF16 + 5, acc, 0, None, None, 1.0, **kw) == 2
    # an owner accumulator overlapping a gradient, an output, or another one
    assert g(table, m, K, 2, 64, B.DP_BF16, acc[:3] + [fake(3, 8)], 0, None, None, 1.0,
             **kw) == 3
    assert g(table, m, K, 2, 64, B.DP_BF16, acc[:3] + [fake(30, 16)], L, outs, None, 1.0,
             **kw) == 3
    assert g(table, m, K, 2, 64, B.DP_BF16, acc[:3] + [fake(20, 16)], 0, None, None, 1.0,
             **kw) == 3
    # outputs are not looked at before the last group (NULL is fine)
    assert g(table, m, K, 2, 0, B.DP_BF16, acc, 0, None, None, 1.0, **kw) == 0
    # one settle for the whole minibatch needs no accumulator
    assert g(table, m, K, 2, 0, B.DP_BF16, None, F | L, outs, None, 1.0, **kw) == 0
    # the pipe: a NULL handle is rejected; create needs a device
    assert B.load().dp_settle_pipe_wait(None, None) == 1
    assert B.load().dp_settle_pipe_destroy(None) == 1
    assert B.dp_settle_pipe_push(0, table, m, K, 2, 64, B.DP_BF16, acc, 0, None, None, 1.0,
                                 **kw) == 1
    assert B.load().dp_settle_pipe_create(-1, ctypes.byref(ctypes.c_void_p())) == 1


def test_the_product_fails_loudly_without_the_library(monkeypatch):
    """No CPU or PyTorch fallback: with the CUDA library missing, the binding
    and the tensor helpers raise instead of computing anything."""
    import torch
    from ring_allreduce_gradient_gb300 import collectives as col
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libdp_gb300.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.load()
    bufs = [torch.ones(16), torch.ones(16)]
    with pytest.raises(RuntimeError, match="missing"):
        col.all_reduce_(bufs, 0.5)
    assert all(bool((b == 1).all()) for b in bufs)
    with pytest.raises(RuntimeError, match="missing"):
        col.reduce_scatter(bufs, 0.5)
