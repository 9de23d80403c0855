// dp_stream.cu -- the HBM-streaming kernels of the ring collectives.
//
// The ring of "CMU 11-868 L14-L15: Distributed Training and Data Parallelism,
// and Where Gradient Sync Costs Come From" (section "Ring AllReduce:
// ReduceScatter, then AllGather") moves chunks between workers in K-1
// reduce-scatter steps and K-1 all-gather steps.  With the K ranks' buffers
// in one GPU's memory none of those hops has to be executed: the steps only
// fix, for each element, the order of its fp32 additions -- chunk c is folded
// x_{c+1} + x_{c+2} + ... + x_{c}.  So each kernel here reads each rank's
// element once, folds in that order in registers, applies the average and the
// output cast, and writes once.  No kernel needs inter-CTA synchronisation.
//
// Layout: grid.y is the chunk index c, so the fold's starting rank and the
// output shard are uniform per CTA; grid.x CTAs stride through the chunk in
// units of 8 elements (one or two 16-byte loads per rank).  The grid is sized
// from the SM count times the kernel's occupancy (a persistent grid-stride
// loop), split evenly across the chunks.
//
// Additions use __fadd_rn and the scale __fmul_rn, so no contraction or
// reassociation can change the ring's rounding.

#include "dp_stream_common.cuh"

namespace {

template <typename T>
__host__ __device__ constexpr int units_per_iter(int kmax) {
  // Keep about thirty-two 16-byte loads in flight per thread.  For the K=8
  // bf16 reduce-scatter on GB300 this is never slower than sixteen (6.56 vs
  // 6.52 TB/s in back-to-back runs; in a state where the same GPU streams
  // about 7% faster the gap widened to 4%).  Twenty-four loses a CTA per SM
  // without adding bytes in flight.
  return (32 / (kmax * Vec8<T>::kLoads)) > 0 ? (32 / (kmax * Vec8<T>::kLoads)) : 1;
}

// ---------------------------------------------------------------------------
// Reduce-scatter
// ---------------------------------------------------------------------------
struct RsParams {
  const void* in[kMaxK];
  float* out32[kMaxK];
  uint16_t* out16[kMaxK];
  int K;
  size_t C;      // chunk length (N / K)
  size_t units;  // C / 8 (vector path)
  float scale;
};

template <typename Tin, int KMAX, bool W32, bool W16>
__global__ void __launch_bounds__(kThreads)
    rs_vec_kernel(const __grid_constant__ RsParams p) {
  constexpr int U = units_per_iter<Tin>(KMAX);
  constexpr int L = Vec8<Tin>::kLoads;
  const int c = blockIdx.y;
  const int K = p.K;
  const size_t chunk0 = (size_t)c * p.C;

  const Tin* src[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    src[j] = (j < K) ? static_cast<const Tin*>(p.in[ring_rank(c, j, K)]) + chunk0 : nullptr;
  float* o32 = W32 ? p.out32[c] : nullptr;
  uint16_t* o16 = W16 ? p.out16[c] : nullptr;

  const size_t T = (size_t)gridDim.x * kThreads;
  for (size_t u0 = (size_t)blockIdx.x * kThreads + threadIdx.x; u0 < p.units; u0 += T * U) {
    uint4 raw[U][KMAX][L];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t u = u0 + (size_t)k * T;
      if (u < p.units) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < K) Vec8<Tin>::load(src[j] + u * 8, raw[k][j]);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t u = u0 + (size_t)k * T;
      if (u < p.units) {
        float acc[8];
        Vec8<Tin>::widen(raw[k][0], acc);
#pragma unroll
        for (int j = 1; j < KMAX; ++j) {
          if (j < K) {
            float v[8];
            Vec8<Tin>::widen(raw[k][j], v);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], v[e]);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fmul_rn(acc[e], p.scale);
        if (W32) store8_f32(o32 + u * 8, acc);
        if (W16) store8_bf16(o16 + u * 8, acc);
      }
    }
  }
}

// Any alignment, any chunk length: one element per thread.
template <typename Tin>
__global__ void __launch_bounds__(kThreads) rs_scalar_kernel(const __grid_constant__ RsParams p) {
  const int c = blockIdx.y;
  const int K = p.K;
  const size_t chunk0 = (size_t)c * p.C;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < p.C;
       i += (size_t)gridDim.x * kThreads) {
    float acc = widen_scalar(static_cast<const Tin*>(p.in[ring_rank(c, 0, K)]), chunk0 + i);
    for (int j = 1; j < K; ++j)
      acc = __fadd_rn(acc, widen_scalar(static_cast<const Tin*>(p.in[ring_rank(c, j, K)]),
                                        chunk0 + i));
    acc = __fmul_rn(acc, p.scale);
    if (p.out32[c]) p.out32[c][i] = acc;
    if (p.out16[c]) p.out16[c][i] = bf16_rn(acc);
  }
}

// ---------------------------------------------------------------------------
// All-reduce (in place): fold, average, cast, and write the same value to
// every rank's buffer.  Chunks are C = ceil(N/K) long; the last may be short.
// ---------------------------------------------------------------------------
struct ArParams {
  void* bufs[kMaxK];
  int K;
  size_t N;
  size_t C;
  float scale;
};

template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&v)[8]) {
  store8_f32(p, v);
}
template <>
__device__ __forceinline__ void store8<uint16_t>(uint16_t* p, const float (&v)[8]) {
  store8_bf16(p, v);
}

__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(uint16_t* p, float v) { *p = bf16_rn(v); }

template <typename T, int KMAX>
__global__ void __launch_bounds__(kThreads) ar_vec_kernel(const __grid_constant__ ArParams p) {
  constexpr int U = units_per_iter<T>(KMAX);
  constexpr int L = Vec8<T>::kLoads;
  const int c = blockIdx.y;
  const int K = p.K;
  const size_t chunk0 = (size_t)c * p.C;
  if (chunk0 >= p.N) return;
  const size_t len = (p.N - chunk0) < p.C ? (p.N - chunk0) : p.C;
  const size_t units = len / 8;

  T* buf[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    buf[j] = (j < K) ? static_cast<T*>(p.bufs[ring_rank(c, j, K)]) + chunk0 : nullptr;

  const size_t Tn = (size_t)gridDim.x * kThreads;
  for (size_t u0 = (size_t)blockIdx.x * kThreads + threadIdx.x; u0 < units; u0 += Tn * U) {
    uint4 raw[U][KMAX][L];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t u = u0 + (size_t)k * Tn;
      if (u < units) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < K) Vec8<T>::load_rw(buf[j] + u * 8, raw[k][j]);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t u = u0 + (size_t)k * Tn;
      if (u < units) {
        float acc[8];
        Vec8<T>::widen(raw[k][0], acc);
#pragma unroll
        for (int j = 1; j < KMAX; ++j) {
          if (j < K) {
            float v[8];
            Vec8<T>::widen(raw[k][j], v);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], v[e]);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fmul_rn(acc[e], p.scale);
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < K) store8<T>(buf[j] + u * 8, acc);
      }
    }
  }
  // ragged tail of a short last chunk (fewer than 8 elements)
  if (blockIdx.x == 0) {
    for (size_t i = units * 8 + threadIdx.x; i < len; i += kThreads) {
      float acc = widen_scalar(static_cast<const T*>(p.bufs[ring_rank(c, 0, K)]), chunk0 + i);
      for (int j = 1; j < K; ++j)
        acc = __fadd_rn(acc, widen_scalar(static_cast<const T*>(p.bufs[ring_rank(c, j, K)]),
                                          chunk0 + i));
      acc = __fmul_rn(acc, p.scale);
      for (int j = 0; j < K; ++j) store1(static_cast<T*>(p.bufs[j]) + chunk0 + i, acc);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) ar_scalar_kernel(const __grid_constant__ ArParams p) {
  const int c = blockIdx.y;
  const int K = p.K;
  const size_t chunk0 = (size_t)c * p.C;
  if (chunk0 >= p.N) return;
  const size_t len = (p.N - chunk0) < p.C ? (p.N - chunk0) : p.C;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < len;
       i += (size_t)gridDim.x * kThreads) {
    float acc = widen_scalar(static_cast<const T*>(p.bufs[ring_rank(c, 0, K)]), chunk0 + i);
    for (int j = 1; j < K; ++j)
      acc = __fadd_rn(acc, widen_scalar(static_cast<const T*>(p.bufs[ring_rank(c, j, K)]),
                                        chunk0 + i));
    acc = __fmul_rn(acc, p.scale);
    for (int j = 0; j < K; ++j) store1(static_cast<T*>(p.bufs[j]) + chunk0 + i, acc);
  }
}

// ---------------------------------------------------------------------------
// All-gather: shard c (rank c's finished chunk) is copied into chunk c of
// every rank's buffer.  A byte copy; 16-byte vectors when everything is
// aligned.  Reads each shard once and writes it K times.
// ---------------------------------------------------------------------------
struct AgParams {
  const unsigned char* shards[kMaxK];
  unsigned char* out[kMaxK];
  int K;
  size_t bytes;  // bytes per shard
  size_t vecs;   // bytes / 16
};

template <int KMAX>
__global__ void __launch_bounds__(kThreads) ag_vec_kernel(const __grid_constant__ AgParams p) {
  constexpr int U = 4;
  const int c = blockIdx.y;
  const int K = p.K;
  const unsigned char* src = p.shards[c];
  const size_t off = (size_t)c * p.bytes;
  unsigned char* dst[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) dst[j] = (j < K) ? p.out[j] + off : nullptr;
  const size_t T = (size_t)gridDim.x * kThreads;
  for (size_t v0 = (size_t)blockIdx.x * kThreads + threadIdx.x; v0 < p.vecs; v0 += T * U) {
    uint4 val[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t v = v0 + (size_t)k * T;
      if (v < p.vecs) val[k] = ld_stream_v4(src + v * 16);
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t v = v0 + (size_t)k * T;
      if (v < p.vecs) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < K) st_stream_v4(dst[j] + v * 16, val[k]);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads) ag_scalar_kernel(const __grid_constant__ AgParams p) {
  const int c = blockIdx.y;
  const unsigned char* src = p.shards[c];
  const size_t off = (size_t)c * p.bytes;
  for (size_t b = (size_t)blockIdx.x * kThreads + threadIdx.x; b < p.bytes;
       b += (size_t)gridDim.x * kThreads) {
    const unsigned char v = src[b];
    for (int j = 0; j < p.K; ++j) p.out[j][off + b] = v;
  }
}

// ---------------------------------------------------------------------------
// Bounded-wait self-test: one thread waits on an mbarrier that nothing will
// complete, gives up after the deadline and flags the error word.
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(unsigned* err_word, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: nobody arrives
    (void)mbar_wait_bounded(&bar, 0u, err_word, timeout_ns);
  }
  __syncthreads();
  if (threadIdx.x == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
}


template <typename Tin, int KMAX>
cudaError_t rs_launch_k(const RsParams& p, bool w32, bool w16, const dph::DeviceInfo& dev,
                        cudaStream_t s) {
  void (*kern)(RsParams);
  if (w32 && w16) kern = rs_vec_kernel<Tin, KMAX, true, true>;
  else if (w32) kern = rs_vec_kernel<Tin, KMAX, true, false>;
  else kern = rs_vec_kernel<Tin, KMAX, false, true>;
  const int occ = occupancy_blocks(kern, dev.device);
  constexpr int U = units_per_iter<Tin>(KMAX);
  dim3 grid(grid_x(dev.sm_count, occ, p.K, p.units, kThreads * U), p.K);
  kern<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t rs_launch_t(const RsParams& p, bool w32, bool w16, bool vec,
                        const dph::DeviceInfo& dev, cudaStream_t s) {
  if (!vec) {
    const int occ = occupancy_blocks(rs_scalar_kernel<Tin>, dev.device);
    dim3 grid(grid_x(dev.sm_count, occ, p.K, p.C, kThreads), p.K);
    rs_scalar_kernel<Tin><<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  switch (kmax_for(p.K)) {
    case 2: return rs_launch_k<Tin, 2>(p, w32, w16, dev, s);
    case 4: return rs_launch_k<Tin, 4>(p, w32, w16, dev, s);
    case 8: return rs_launch_k<Tin, 8>(p, w32, w16, dev, s);
    default: return rs_launch_k<Tin, 16>(p, w32, w16, dev, s);
  }
}

template <typename T, int KMAX>
cudaError_t ar_launch_k(const ArParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  const int occ = occupancy_blocks(ar_vec_kernel<T, KMAX>, dev.device);
  constexpr int U = units_per_iter<T>(KMAX);
  dim3 grid(grid_x(dev.sm_count, occ, p.K, p.C / 8 + 1, kThreads * U), p.K);
  ar_vec_kernel<T, KMAX><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t ar_launch_t(const ArParams& p, bool vec, const dph::DeviceInfo& dev, cudaStream_t s) {
  if (!vec) {
    const int occ = occupancy_blocks(ar_scalar_kernel<T>, dev.device);
    dim3 grid(grid_x(dev.sm_count, occ, p.K, p.C, kThreads), p.K);
    ar_scalar_kernel<T><<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  switch (kmax_for(p.K)) {
    case 2: return ar_launch_k<T, 2>(p, dev, s);
    case 4: return ar_launch_k<T, 4>(p, dev, s);
    case 8: return ar_launch_k<T, 8>(p, dev, s);
    default: return ar_launch_k<T, 16>(p, dev, s);
  }
}

template <int KMAX>
cudaError_t ag_launch_k(const AgParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  const int occ = occupancy_blocks(ag_vec_kernel<KMAX>, dev.device);
  dim3 grid(grid_x(dev.sm_count, occ, p.K, p.vecs, kThreads * 4), p.K);
  ag_vec_kernel<KMAX><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

namespace dpl {

cudaError_t launch_reduce_scatter(const RsArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  RsParams p{};
  for (int r = 0; r < a.K; ++r) {
    p.in[r] = a.in[r];
    p.out32[r] = a.out32[r];
    p.out16[r] = a.out16[r];
  }
  p.K = a.K;
  p.C = a.C;
  p.units = a.C / 8;
  p.scale = a.scale;
  const bool w32 = a.out32[0] != nullptr, w16 = a.out16[0] != nullptr;
  if (a.in_dtype == DP_FP32) return rs_launch_t<float>(p, w32, w16, a.vec_ok, dev, s);
  return rs_launch_t<uint16_t>(p, w32, w16, a.vec_ok, dev, s);
}

cudaError_t launch_all_gather(const AgArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  AgParams p{};
  for (int r = 0; r < a.K; ++r) {
    p.shards[r] = static_cast<const unsigned char*>(a.shards[r]);
    p.out[r] = static_cast<unsigned char*>(a.out[r]);
  }
  p.K = a.K;
  p.bytes = a.C * a.esz;
  p.vecs = p.bytes / 16;
  if (!a.vec_ok) {
    const int occ = occupancy_blocks(ag_scalar_kernel, dev.device);
    dim3 grid(grid_x(dev.sm_count, occ, p.K, p.bytes, kThreads), p.K);
    ag_scalar_kernel<<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  switch (kmax_for(a.K)) {
    case 2: return ag_launch_k<2>(p, dev, s);
    case 4: return ag_launch_k<4>(p, dev, s);
    case 8: return ag_launch_k<8>(p, dev, s);
    default: return ag_launch_k<16>(p, dev, s);
  }
}

cudaError_t launch_all_reduce(const ArArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  ArParams p{};
  for (int r = 0; r < a.K; ++r) p.bufs[r] = a.bufs[r];
  p.K = a.K;
  p.N = a.N;
  p.C = a.C;
  p.scale = a.scale;
  if (a.dtype == DP_FP32) return ar_launch_t<float>(p, a.vec_ok, dev, s);
  return ar_launch_t<uint16_t>(p, a.vec_ok, dev, s);
}

cudaError_t launch_selftest_wait(uint32_t timeout_us, const dph::DeviceInfo& dev, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(dev.err_word, (uint64_t)timeout_us * 1000ull);
  return cudaGetLastError();
}

}  // namespace dpl
