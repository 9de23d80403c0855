"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays them out; it holds none of the
collective's arithmetic (no fold, no average, no output cast), so both the
CUDA path's tests and the oracle may take their inputs from it.

Recipes (the pages use models and data that are not available here, so these
synthetic tensors stand in for "a rank's gradient" and "a layer's weights"):

* ``ring_ints``     -- K=4 ranks, N=4096 fp32, integers uniform in {-8..8},
  per-rank stream ``SeedSequence(0).spawn(K)[r]``.  Every partial sum is an
  integer of magnitude <= 32, so every summation order is exact.
* ``fsdp_grads``    -- K ranks of N bf16 gradients, N(0, 1e-3) (1e-3 is the
  standard deviation) drawn in fp32 with seed r, then rounded to bf16 (RNE,
  by PyTorch's conversion).
* ``sweep_bufs``    -- K ranks of N fp32 values uniform in [-1, 1], seed
  1000*K + r.
* ``gemm_operands`` -- x[M, D] and K row shards w_k[F_shard, D] in bf16,
  N(0, 0.02), seeds 40 (x) and 41+k (w_k).
* ``odc_schedule`` / ``odc_grad`` -- K=8 ranks, microbatch counts m_r uniform
  in 1..8 (seed 5), token counts per microbatch lognormal with median 1024,
  sigma 1.0, rounded and clamped to [1, 8192] (seed 6); the gradient of
  microbatch j of rank r in layer l is N(0, 1e-3) * t_{r,j} rounded to bf16,
  from a generator seeded with ``odc_seed(l, r, j)``.

bf16 values are returned as raw 16-bit patterns in ``numpy.uint16`` arrays on
the host, or as ``torch.bfloat16`` tensors where a device is requested.
"""
from __future__ import annotations

import math

import numpy as np
import torch

MiB = 1 << 20


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (PyTorch's round-to-nearest-even conversion), as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_torch_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


def ring_ints(K: int = 4, N: int = 4096, seed: int = 0) -> list[np.ndarray]:
    seqs = np.random.SeedSequence(seed).spawn(K)
    return [np.random.default_rng(s).integers(-8, 9, size=N).astype(np.float32) for s in seqs]


def fsdp_grads(K: int = 8, N: int = 64 * MiB, std: float = 1e-3) -> list[np.ndarray]:
    out = []
    for r in range(K):
        g = np.random.default_rng(r).standard_normal(N, dtype=np.float32)
        g *= np.float32(std)
        out.append(to_bf16_bits(g))
    return out


def fsdp_grads_device(K: int, N: int, device, std: float = 1e-3) -> list[torch.Tensor]:
    """The same recipe drawn on a device with PyTorch's generator (seed r)."""
    out = []
    for r in range(K):
        g = torch.Generator(device=device)
        g.manual_seed(r)
        t = torch.randn(N, generator=g, device=device, dtype=torch.float32)
        out.append((t * std).to(torch.bfloat16))
    return out


def sweep_bufs(K: int, N: int) -> list[np.ndarray]:
    return [np.random.default_rng(1000 * K + r).uniform(-1.0, 1.0, N).astype(np.float32)
            for r in range(K)]


def sweep_bufs_device(K: int, N: int, device) -> list[torch.Tensor]:
    out = []
    for r in range(K):
        g = torch.Generator(device=device)
        g.manual_seed(1000 * K + r)
        out.append(torch.rand(N, generator=g, device=device, dtype=torch.float32) * 2 - 1)
    return out


def sweep_sizes_bytes() -> list[int]:
    """Per-rank buffer sizes of the bandwidth sweep: 4 KiB .. 1 GiB in x4 steps."""
    return [4096 * 4 ** n for n in range(10)]


def gemm_operands(M: int, D: int, K: int, F_shard: int, std: float = 0.02):
    rx = np.random.default_rng(40)
    x = to_bf16_bits(rx.standard_normal((M, D), dtype=np.float32) * np.float32(std))
    ws = []
    for k in range(K):
        rw = np.random.default_rng(41 + k)
        ws.append(to_bf16_bits(rw.standard_normal((F_shard, D), dtype=np.float32) *
                               np.float32(std)))
    return x, ws


def gemm_int_operands(M: int, D: int, K: int, F_shard: int, seed: int = 7):
    """Integer-valued bf16 operands in [-4, 4]: with D <= 512 every fp32
    partial sum is an integer below 2^24, so the product is exact."""
    rng = np.random.default_rng(seed)
    x = to_bf16_bits(rng.integers(-4, 5, (M, D)).astype(np.float32))
    ws = [to_bf16_bits(rng.integers(-4, 5, (F_shard, D)).astype(np.float32)) for _ in range(K)]
    return x, ws


def tp_operands(M: int, D_shard: int, F: int, K: int, std: float = 0.02, ints: bool = False):
    """Tensor-parallel partial-dot operands: rank r holds x_r [M, D_shard] and
    w_r [F, D_shard] (weight in the [out, in] layout), bf16 N(0, std) (seeds
    60+r, 80+r), or integers in [-4, 4] when ``ints``."""
    xs, ws = [], []
    for r in range(K):
        rx, rw = np.random.default_rng(60 + r), np.random.default_rng(80 + r)
        if ints:
            xs.append(to_bf16_bits(rx.integers(-4, 5, (M, D_shard)).astype(np.float32)))
            ws.append(to_bf16_bits(rw.integers(-4, 5, (F, D_shard)).astype(np.float32)))
        else:
            xs.append(to_bf16_bits(rx.standard_normal((M, D_shard), dtype=np.float32) *
                                   np.float32(std)))
            ws.append(to_bf16_bits(rw.standard_normal((F, D_shard), dtype=np.float32) *
                                   np.float32(std)))
    return xs, ws


def wgrad_operands(T: int, F: int, D: int, K: int, std: float = 0.02, ints: bool = False):
    """Weight-gradient operands of a linear layer y = x . w^T on K ranks: rank r
    holds dy_r [T, F] (output gradients) and x_r [T, D] (inputs), tokens x
    features, bf16 N(0, std) (seeds 90+r, 110+r), or integers in [-4, 4] when
    ``ints``."""
    dys, xs = [], []
    for r in range(K):
        rd, rx = np.random.default_rng(90 + r), np.random.default_rng(110 + r)
        if ints:
            dys.append(to_bf16_bits(rd.integers(-4, 5, (T, F)).astype(np.float32)))
            xs.append(to_bf16_bits(rx.integers(-4, 5, (T, D)).astype(np.float32)))
        else:
            dys.append(to_bf16_bits(rd.standard_normal((T, F), dtype=np.float32) *
                                    np.float32(std)))
            xs.append(to_bf16_bits(rx.standard_normal((T, D), dtype=np.float32) *
                                   np.float32(std)))
    return dys, xs


def gpt2_small_numels(layers: int = 12, d: int = 768, vocab: int = 50257, ctx: int = 1024):
    """Parameter sizes of a GPT-2-small-shaped model (124,439,808 parameters in
    148 tensors), in model.parameters() order."""
    out = [vocab * d, ctx * d]
    for _ in range(layers):
        out += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    out += [d, d]
    return out


def ddp_grads_device(numels, K: int, device):
    """fp32 gradients U[-1, 1] of every parameter on K ranks, drawn on the
    device (CUDA generator seeded 700 + r, tensors in parameter order)."""
    grads = [[torch.empty(n, device=device) for n in numels] for _ in range(K)]
    for r in range(K):
        g = torch.Generator(device=device)
        g.manual_seed(700 + r)
        for t in grads[r]:
            t.uniform_(-1, 1, generator=g)
    return grads


def odc_schedule(K: int = 8, max_mb: int = 8, median_tokens: int = 1024, sigma: float = 1.0,
                 cap: int = 8192):
    """Microbatch counts m_r and token counts t[r][j] of the variable-length step."""
    m = np.random.default_rng(5).integers(1, max_mb + 1, size=K)
    rt = np.random.default_rng(6)
    z = rt.standard_normal((K, max_mb))
    t = np.clip(np.rint(np.exp(math.log(median_tokens) + sigma * z)), 1, cap).astype(np.int64)
    return [int(v) for v in m], t


def odc_seed(layer: int, r: int, j: int) -> int:
    return 6_000_000 + 10_000 * layer + 100 * r + j


def odc_grad(layer: int, r: int, j: int, N: int, tokens: int, device="cpu",
             std: float = 1e-3) -> torch.Tensor:
    """One microbatch gradient (bf16 tensor on ``device``)."""
    g = torch.Generator(device=device)
    g.manual_seed(odc_seed(layer, r, j))
    t = torch.randn(N, generator=g, device=device, dtype=torch.float32)
    return (t * std * float(tokens)).to(torch.bfloat16)


def torch_bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
