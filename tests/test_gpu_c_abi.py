"""The C ABI used from plain C: a small program includes include/dp.h, links
libdp_gb300.so and the CUDA runtime, allocates with cudaMalloc and checks the
all-reduce and reduce-scatter against exact integer sums -- no Python or
PyTorch between the caller and the library."""
import os
import subprocess

import pytest

from ring_allreduce_gradient_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "dp.h"

#define K 4
#define N 4096

int main(void) {
  float* host[K];
  void* dev[K];
  void* shards[K];
  float expect[N];
  unsigned seed = 12345u;
  for (int e = 0; e < N; ++e) expect[e] = 0.0f;
  for (int r = 0; r < K; ++r) {
    host[r] = (float*)malloc(N * sizeof(float));
    for (int e = 0; e < N; ++e) {
      seed = seed * 1103515245u + 12345u;
      host[r][e] = (float)((int)((seed >> 16) % 17u) - 8);  /* integers in [-8, 8] */
      expect[e] += host[r][e];
    }
    if (cudaMalloc(&dev[r], N * sizeof(float)) != cudaSuccess) return 10;
    if (cudaMalloc(&shards[r], (N / K) * sizeof(float)) != cudaSuccess) return 11;
    cudaMemcpy(dev[r], host[r], N * sizeof(float), cudaMemcpyHostToDevice);
  }
  /* reduce-scatter into fp32 shards, then all-reduce in place */
  dp_status_t st = dp_reduce_scatter((const void* const*)dev, K, N, DP_FP32, shards, 1.0f,
                                     DP_FP32, (dp_stream_t)0);
  if (st != DP_OK) { printf("rs: %s\n", dp_status_string(st)); return 12; }
  st = dp_ring_allreduce(dev, K, N, DP_FP32, 1.0f, (dp_stream_t)0);
  if (st != DP_OK) { printf("ar: %s\n", dp_status_string(st)); return 13; }
  if (dp_get_device_error((dp_stream_t)0) != DP_OK) return 14;
  float out[N];
  for (int r = 0; r < K; ++r) {
    cudaMemcpy(out, dev[r], N * sizeof(float), cudaMemcpyDeviceToHost);
    for (int e = 0; e < N; ++e)
      if (out[e] != expect[e]) { printf("ar mismatch r=%d e=%d\n", r, e); return 15; }
    cudaMemcpy(out, shards[r], (N / K) * sizeof(float), cudaMemcpyDeviceToHost);
    for (int i = 0; i < N / K; ++i)
      if (out[i] != expect[r * (N / K) + i]) { printf("rs mismatch c=%d i=%d\n", r, i); return 16; }
  }
  /* an invalid call is rejected with a status, not a crash */
  if (dp_ring_allreduce(dev, 0, N, DP_FP32, 1.0f, (dp_stream_t)0) != DP_ERR_INVALID_ARG) return 17;

  /* the settle pipeline: rank r has m[r] microbatches g_{r,j} = (j+1) * x_r
   * (integer-valued, so every order is exact), settled in two groups
   * (j < 1, j >= 1) on the pipe's stream and joined once */
  {
    const int m[K] = {2, 1, 3, 2};
    void* g[K][3];
    float* acc[K];
    float* o32[K];
    float tmp[N];
    for (int r = 0; r < K; ++r) {
      for (int j = 0; j < m[r]; ++j) {
        for (int e = 0; e < N; ++e) tmp[e] = host[r][e] * (float)(j + 1);
        if (cudaMalloc(&g[r][j], N * sizeof(float)) != cudaSuccess) return 20;
        cudaMemcpy(g[r][j], tmp, N * sizeof(float), cudaMemcpyHostToDevice);
      }
      if (cudaMalloc((void**)&acc[r], (N / K) * sizeof(float)) != cudaSuccess) return 21;
      if (cudaMalloc((void**)&o32[r], (N / K) * sizeof(float)) != cudaSuccess) return 22;
    }
    cudaStream_t s;
    if (cudaStreamCreate(&s) != cudaSuccess) return 23;
    dp_settle_pipe_t* pipe = NULL;
    if (dp_settle_pipe_create(0, &pipe) != DP_OK) return 24;
    const void* t0[K];          /* group 0: microbatch 0 of every rank */
    int m0[K];
    const void* t1[K * 2];      /* group 1: microbatches 1 and 2 (K x 2 table) */
    int m1[K];
    for (int r = 0; r < K; ++r) {
      t0[r] = g[r][0];
      m0[r] = 1;
      m1[r] = m[r] - 1;
      t1[2 * r] = m[r] > 1 ? g[r][1] : NULL;
      t1[2 * r + 1] = m[r] > 2 ? g[r][2] : NULL;
    }
    if (dp_settle_pipe_push(pipe, t0, m0, K, 1, N, DP_FP32, acc, DP_SETTLE_FIRST, NULL, NULL,
                            1.0f, (dp_stream_t)s) != DP_OK) return 25;
    if (dp_settle_pipe_push(pipe, t1, m1, K, 2, N, DP_FP32, acc, DP_SETTLE_LAST, o32, NULL,
                            1.0f, (dp_stream_t)s) != DP_OK) return 26;
    if (dp_settle_pipe_wait(pipe, (dp_stream_t)s) != DP_OK) return 27;
    if (dp_get_device_error((dp_stream_t)s) != DP_OK) return 28;
    for (int c = 0; c < K; ++c) {
      cudaMemcpy(out, o32[c], (N / K) * sizeof(float), cudaMemcpyDeviceToHost);
      for (int i = 0; i < N / K; ++i) {
        const int e = c * (N / K) + i;
        float want = 0.0f;
        for (int r = 0; r < K; ++r)
          for (int j = 0; j < m[r]; ++j) want += host[r][e] * (float)(j + 1);
        if (out[i] != want) { printf("pipe mismatch c=%d i=%d\n", c, i); return 29; }
      }
    }
    if (dp_settle_pipe_destroy(pipe) != DP_OK) return 30;
  }
  printf("c-abi ok (version %d)\n", dp_version());
  return 0;
}
"""


def test_c_program_links_and_runs(tmp_path):
    lib = cuda_build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c99", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-ldp_gb300", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c-abi ok" in r.stdout
