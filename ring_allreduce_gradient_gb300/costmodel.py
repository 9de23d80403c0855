"""Byte and time accounting for the ring collectives and for this library's
kernels.

Two different byte counts appear here and must not be confused:

* Ring transport bytes -- what one rank sends over its link in a real ring
  of X devices.  "Sharding and Parallelism" (How to Scale Your Model on AMD,
  ch. 5), section "The cost of the inserted collectives":
  T_AG,ring >= B(X-1)/(XW), T_RS,ring >= B(X-1)/(XW),
  T_AR,ring >= 2B(X-1)/(XW), with B the size of the completed all-gather
  buffer (equivalently the reducible buffer of the reduce-scatter) and W
  the achieved one-direction link bandwidth.  The ring broadcast terms come
  from "CMU 11-868 L14-L15 ...", section "Why a ring: chop the data so
  transfers pipeline": (K-1)N/B whole, (K-2+S)N/(SB) in S pieces.
  These are context: the virtual ranks here share one GPU's memory.

* Algorithmic HBM bytes -- the minimum bytes one call of a kernel here must
  read and write in device memory.  Achieved bandwidth is these bytes over
  the kernel's time, and the roofline fraction is that over the measured
  copy bandwidth.
"""
from __future__ import annotations

ELEM = {"f32": 4, "bf16": 2}


# --- ring transport (the pages' cost model) --------------------------------

def ring_allgather_bytes_per_rank(B: float, X: int) -> float:
    """Bytes each rank sends in a ring all-gather of a B-byte result."""
    return B * (X - 1) / X


def ring_reduce_scatter_bytes_per_rank(B: float, X: int) -> float:
    return B * (X - 1) / X


def ring_allreduce_bytes_per_rank(B: float, X: int) -> float:
    return 2.0 * B * (X - 1) / X


def transport_time_s(bytes_sent: float, W_bytes_per_s: float) -> float:
    return bytes_sent / W_bytes_per_s


def ring_broadcast_time_s(K: int, N_bytes: float, B_bytes_per_s: float, S: int = 1) -> float:
    """(K-2+S) N/(S B); S=1 gives the whole-message (K-1) N / B."""
    return (K - 2 + S) * N_bytes / (S * B_bytes_per_s)


# --- algorithmic HBM bytes / flops of one call ------------------------------

def reduce_scatter_hbm_bytes(K: int, N: int, in_dtype: str, out_dtypes) -> int:
    """Read every rank's N elements once; write N output elements per output type."""
    return K * N * ELEM[in_dtype] + sum(N * ELEM[d] for d in out_dtypes)


def all_gather_hbm_bytes(K: int, C: int, dtype: str) -> int:
    """Read the K shards (K*C elements) once; write K buffers of K*C."""
    N = K * C
    return N * ELEM[dtype] + K * N * ELEM[dtype]


def all_reduce_hbm_bytes(K: int, N: int, dtype: str) -> int:
    """In place: read and write every rank's N elements once."""
    return 2 * K * N * ELEM[dtype]


def accumulate_hbm_bytes(N: int, grad_dtype: str, first: bool, pad: bool = False) -> int:
    """acc = (first ? +0 : acc) + g.  A padding bucket reads no gradient."""
    g = 0 if pad else N * ELEM[grad_dtype]
    a_read = 0 if first else N * 4
    return g + a_read + N * 4


def odc_fused_hbm_bytes(total_microbatches: int, N: int, grad_dtype: str, out_dtypes) -> int:
    """One pass: read every real microbatch gradient once, write the shards."""
    return total_microbatches * N * ELEM[grad_dtype] + sum(N * ELEM[d] for d in out_dtypes)


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def allgather_matmul_min_bytes(M: int, D: int, F: int, y_dtype: str = "bf16") -> int:
    return M * D * 2 + F * D * 2 + M * F * ELEM[y_dtype]
