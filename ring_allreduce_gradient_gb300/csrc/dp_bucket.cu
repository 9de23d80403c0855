// dp_bucket.cu -- all-reduce of a DDP gradient bucket, in place, without
// flattening.
//
// "CMU 11-868 L14-L15: Distributed Training and Data Parallelism, and Where
// Gradient Sync Costs Come From", section "When to sync: gradient bucketing":
// gradients are grouped into buckets and each bucket is all-reduced as one
// message.  A ring all-reduce of a bucket treats the bucket as one flat
// buffer of `total` elements split into K chunks of C = ceil(total/K), so the
// fold order of an element depends on its offset inside the bucket.  This
// kernel reads each gradient tensor where it lives (no copy into a flat
// bucket buffer and back), computes every element's bucket offset, folds the
// K ranks' values in that chunk's ring order (x_{c+1} + ... + x_c, fp32),
// scales, casts and writes the result back into all K ranks' tensors.
//
// Work split: tensor t of a launch owns units [ustart[t], ustart[t+1]) of 8
// elements; a grid-stride loop over units finds its tensor by binary search.
// A full unit whose K pointers are 16-byte aligned and whose 8 elements share
// one chunk takes the vector path; anything else (a ragged tail, a chunk
// boundary inside the unit, unaligned tensors) folds element by element with
// the same arithmetic.

#include "dp_launch.h"

#include <algorithm>

namespace {

using namespace dpk;

constexpr int kThreads = 256;
constexpr int kMtMax = 96;  // tensors per launch (kernel parameter space)

struct MtParams {
  void* ptr[kMtMax][kMaxK];
  unsigned long long off[kMtMax];  // bucket offset of the tensor's first element
  unsigned long long numel[kMtMax];
  unsigned ustart[kMtMax + 1];     // prefix sums of units (8 elements) per tensor
  unsigned vec_ok[kMtMax];         // all K pointers 16-byte aligned
  int n, K;
  unsigned long long C;            // chunk length of the whole bucket
  float scale;
};

__device__ __forceinline__ int ring_rank(int c, int j, int K) {
  int r = c + 1 + j;
  return r >= K ? r - K : r;
}

__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(uint16_t* p, float v) { *p = bf16_rn(v); }

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

template <typename T, int KMAX>
__global__ void __launch_bounds__(kThreads) mt_ar_kernel(const __grid_constant__ MtParams p) {
  constexpr int L = Vec8<T>::kLoads;
  const int K = p.K;
  const unsigned total_units = p.ustart[p.n];
  for (unsigned u = blockIdx.x * kThreads + threadIdx.x; u < total_units;
       u += gridDim.x * kThreads) {
    // tensor of this unit: the last t with ustart[t] <= u
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.ustart[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    const int t = lo;
    const unsigned long long e0 = (unsigned long long)(u - p.ustart[t]) * 8ull;
    const unsigned long long len =
        (p.numel[t] - e0) < 8ull ? (p.numel[t] - e0) : 8ull;
    const unsigned long long b0 = p.off[t] + e0;  // bucket offset of the first element
    int c0, c1;
    if (p.C <= 0xffffffffull && b0 + len <= 0xffffffffull) {  // 32-bit division suffices
      c0 = (int)((unsigned)b0 / (unsigned)p.C);
      c1 = (int)((unsigned)(b0 + len - 1) / (unsigned)p.C);
    } else {
      c0 = (int)(b0 / p.C);
      c1 = (int)((b0 + len - 1) / p.C);
    }
    if (len == 8 && c0 == c1 && p.vec_ok[t]) {
      uint4 raw[KMAX][L];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < K) Vec8<T>::load_rw(static_cast<const T*>(p.ptr[t][ring_rank(c0, j, K)]) + e0,
                                    raw[j]);
      float acc[8];
      Vec8<T>::widen(raw[0], acc);
#pragma unroll
      for (int j = 1; j < KMAX; ++j) {
        if (j < K) {
          float v[8];
          Vec8<T>::widen(raw[j], v);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], v[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = __fmul_rn(acc[e], p.scale);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < K) store8<T>(static_cast<T*>(p.ptr[t][j]) + e0, acc);
    } else {
      for (unsigned long long i = 0; i < len; ++i) {
        const int c = (int)((b0 + i) / p.C);
        float acc = widen_scalar(static_cast<const T*>(p.ptr[t][ring_rank(c, 0, K)]), e0 + i);
        for (int j = 1; j < K; ++j)
          acc = __fadd_rn(acc, widen_scalar(static_cast<const T*>(p.ptr[t][ring_rank(c, j, K)]),
                                            e0 + i));
        acc = __fmul_rn(acc, p.scale);
        for (int j = 0; j < K; ++j) store1(static_cast<T*>(p.ptr[t][j]) + e0 + i, acc);
      }
    }
  }
}

template <typename KernelT>
int occupancy_blocks(KernelT kernel, int device) {
  const int b = dph::prepare_kernel(reinterpret_cast<const void*>(kernel), kThreads, 0, device);
  return b < 1 ? 1 : b;
}

template <typename T, int KMAX>
cudaError_t mt_launch_k(const MtParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  const int occ = occupancy_blocks(mt_ar_kernel<T, KMAX>, dev.device);
  const unsigned units = p.ustart[p.n];
  long long resident = (long long)dev.sm_count * occ;
  const int limit = dph::stream_cta_limit();
  if (limit > 0 && resident > limit) resident = limit;
  long long blocks = std::min<long long>(resident, ((long long)units + kThreads - 1) / kThreads);
  if (blocks < 1) blocks = 1;
  mt_ar_kernel<T, KMAX><<<(unsigned)blocks, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t mt_launch_t(const MtParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  const int K = p.K;
  if (K <= 2) return mt_launch_k<T, 2>(p, dev, s);
  if (K <= 4) return mt_launch_k<T, 4>(p, dev, s);
  if (K <= 8) return mt_launch_k<T, 8>(p, dev, s);
  return mt_launch_k<T, 16>(p, dev, s);
}

}  // namespace

namespace dpl {

cudaError_t launch_bucket_allreduce(const BucketArgs& a, const dph::DeviceInfo& dev,
                                    cudaStream_t s) {
  // bucket offsets and the chunk length come from the whole bucket
  unsigned long long total = 0;
  for (int t = 0; t < a.n; ++t) total += a.numels[t];
  if (total == 0) return cudaSuccess;
  const unsigned long long C = (total + (unsigned long long)a.K - 1) / (unsigned long long)a.K;
  unsigned long long off = 0;
  int t = 0;
  while (t < a.n) {
    MtParams p;
    memset(&p, 0, sizeof p);
    p.K = a.K;
    p.C = C;
    p.scale = a.scale;
    int n = 0;
    unsigned units = 0;
    // up to kMtMax tensors, and few enough units to index with 32 bits
    while (t < a.n && n < kMtMax) {
      const unsigned long long ne = a.numels[t];
      const unsigned long long tu = (ne + 7) / 8;
      if (n > 0 && (unsigned long long)units + tu > 0x7fffffffull) break;
      bool al = true;
      for (int r = 0; r < a.K; ++r) {
        p.ptr[n][r] = a.ptrs[(size_t)t * a.K + r];
        al = al && ((reinterpret_cast<uintptr_t>(p.ptr[n][r]) & 15u) == 0);
      }
      p.off[n] = off;
      p.numel[n] = ne;
      p.vec_ok[n] = al ? 1u : 0u;
      p.ustart[n] = units;
      units += (unsigned)tu;
      off += ne;
      ++n;
      ++t;
    }
    p.n = n;
    p.ustart[n] = units;
    if (units > 0) {
      cudaError_t e = a.dtype == DP_FP32 ? mt_launch_t<float>(p, dev, s)
                                         : mt_launch_t<uint16_t>(p, dev, s);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace dpl
