// dp_api.cu -- the extern "C" entry points of include/dp.h: argument
// validation, overlap checks, per-device launch information, the device error
// word, and dispatch to the kernel launchers.  Nothing here computes on the
// host; every step of the data path runs in the kernels.

#include "dp_launch.h"

#include <atomic>
#include <map>
#include <mutex>
#include <stdint.h>
#include <utility>

// The device error word: bounded waits that expire set bits here.  One per
// device (a __device__ variable is instantiated in every context).
__device__ unsigned g_dp_error_word = 0u;

namespace dph {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};
}  // namespace

namespace {
std::atomic<int> g_gemm_cta_limit{0};
std::atomic<int> g_stream_cta_limit{0};
std::atomic<int> g_variant{0};
}  // namespace

int prepare_kernel(const void* kernel, int threads, size_t smem, int device) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, device);
  auto it = done.find(key);
  if (it != done.end()) return it->second;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (b < 1) b = 1;
  done[key] = b;
  return b;
}

int collective_variant() { return g_variant.load(std::memory_order_relaxed); }
void set_collective_variant(int v) { g_variant.store(v, std::memory_order_relaxed); }

int gemm_cta_limit() { return g_gemm_cta_limit.load(std::memory_order_relaxed); }
int stream_cta_limit() { return g_stream_cta_limit.load(std::memory_order_relaxed); }
void set_cta_limits(int g, int s) {
  g_gemm_cta_limit.store(g, std::memory_order_relaxed);
  g_stream_cta_limit.store(s, std::memory_order_relaxed);
}

bool current_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev_ready[dev]) {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    d.sm_count = v;
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.smem_optin = (size_t)v;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dp_error_word) != cudaSuccess || !p) {
      cudaGetLastError();
      return false;
    }
    d.err_word = static_cast<unsigned*>(p);
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  *out = g_dev[dev];
  return true;
}

}  // namespace dph

namespace {

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Range& a, const Range& b) {
  return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo;
}

// True if any two ranges of `w` overlap, or any range of `w` overlaps one of `r`.
bool any_overlap(const Range* w, int nw, const Range* r, int nr) {
  for (int i = 0; i < nw; ++i) {
    for (int j = i + 1; j < nw; ++j)
      if (overlaps(w[i], w[j])) return true;
    for (int j = 0; j < nr; ++j)
      if (overlaps(w[i], r[j])) return true;
  }
  return false;
}

Range range_of(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}

size_t dtype_size(dp_dtype_t t) { return t == DP_FP32 ? 4u : 2u; }
bool dtype_ok(dp_dtype_t t) { return t == DP_FP32 || t == DP_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dp_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? DP_OK : DP_ERR_CUDA; }

// Whether the all-reduce / all-gather take the bulk-copy (shared-memory
// staged) kernels; both variants give identical bits.
bool use_bulk_copy() {
  const int v = dph::collective_variant();
  return v == dph::kVariantBulkCopy || v == dph::kVariantAuto;
}

// The automatic choice for the all-reduce: below 32 KiB per rank a call is
// all start-up, and the register kernel starts faster (measured on GB300,
// K=8: 6.1 against 7.2-8.2 us at 4-16 KiB per rank; equal from 64 KiB up).
bool all_reduce_bulk(size_t bytes_per_rank) {
  const int v = dph::collective_variant();
  if (v == dph::kVariantAuto) return bytes_per_rank > 32768;
  return v == dph::kVariantBulkCopy;
}

}  // namespace

namespace dph {

// Validation shared by the one-settle call, the group settle and the settle
// pipeline.  Fills *a (cta_limit 0) or returns the error; *noop is set for
// N == 0, where nothing is launched.
dp_status_t odc_prepare(const void* const* grads, const int* m, int K, int Mmax, size_t N,
                        dp_dtype_t grad_dtype, float* const* owner_acc, int phase,
                        float* const* out_f32, void* const* out_bf16, float scale,
                        dpl::OdcArgs* a, bool* noop) {
  *noop = false;
  if (!grads || !m || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (Mmax < 0 || Mmax > DP_MAX_MICROBATCHES) return DP_ERR_INVALID_ARG;
  if (phase & ~(DP_SETTLE_FIRST | DP_SETTLE_LAST)) return DP_ERR_INVALID_ARG;
  const bool last = (phase & DP_SETTLE_LAST) != 0;
  const bool need_acc = phase != (DP_SETTLE_FIRST | DP_SETTLE_LAST);
  if (last && !out_f32 && !out_bf16) return DP_ERR_INVALID_ARG;
  if (need_acc && !owner_acc) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(grad_dtype)) return DP_ERR_UNSUPPORTED;
  if (N % (size_t)K) return DP_ERR_INVALID_ARG;
  if (!last) {  // outputs unused before the last group
    out_f32 = nullptr;
    out_bf16 = nullptr;
  }
  const size_t C = N / (size_t)K;
  const size_t gsz = dtype_size(grad_dtype);
  Range rin[DP_MAX_K * DP_MAX_MICROBATCHES], rout[3 * DP_MAX_K];
  int nin = 0, nout = 0;
  bool vec = (C % 8) == 0;
  for (int r = 0; r < K; ++r) {
    if (m[r] < 0 || m[r] > Mmax) return DP_ERR_INVALID_ARG;
    if (out_f32 && !out_f32[r]) return DP_ERR_INVALID_ARG;
    if (out_bf16 && !out_bf16[r]) return DP_ERR_INVALID_ARG;
    if (need_acc && !owner_acc[r]) return DP_ERR_INVALID_ARG;
    for (int j = 0; j < m[r]; ++j) {
      const void* g = grads[(size_t)r * Mmax + j];
      if (g) {
        rin[nin++] = range_of(g, N * gsz);
        vec = vec && aligned16(g);
      }
    }
    if (out_f32) rout[nout++] = range_of(out_f32[r], C * 4);
    if (out_bf16) rout[nout++] = range_of(out_bf16[r], C * 2);
    if (need_acc) rout[nout++] = range_of(owner_acc[r], C * 4);
    vec = vec && (!out_f32 || aligned16(out_f32[r])) && (!out_bf16 || aligned16(out_bf16[r])) &&
          (!need_acc || aligned16(owner_acc[r]));
  }
  if (N == 0) {
    *noop = true;
    return DP_OK;
  }
  if (any_overlap(rout, nout, rin, nin)) return DP_ERR_ALIAS;
  *a = dpl::OdcArgs{};
  for (int r = 0; r < K; ++r) {
    for (int j = 0; j < m[r]; ++j) a->grads[r][j] = grads[(size_t)r * Mmax + j];
    a->m[r] = m[r];
    a->out32[r] = out_f32 ? out_f32[r] : nullptr;
    a->out16[r] = out_bf16 ? static_cast<uint16_t*>(out_bf16[r]) : nullptr;
    a->carry[r] = need_acc ? owner_acc[r] : nullptr;
  }
  a->phase = phase;
  a->K = K;
  a->N = N;
  a->C = C;
  a->scale = scale;
  a->grad_dtype = grad_dtype;
  a->vec_ok = vec;
  return DP_OK;
}

dp_status_t odc_launch(const dpl::OdcArgs& a, cudaStream_t s) {
  DeviceInfo dev;
  if (!current_device(&dev)) return DP_ERR_CUDA;
  const cudaError_t e = dpl::launch_odc_reduce_scatter(a, dev, s);
  if (e != cudaSuccess) return DP_ERR_CUDA;
  return DP_OK;
}

}  // namespace dph

extern "C" {

const char* dp_status_string(dp_status_t s) {
  switch (s) {
    case DP_OK: return "DP_OK";
    case DP_ERR_INVALID_ARG: return "DP_ERR_INVALID_ARG";
    case DP_ERR_UNSUPPORTED: return "DP_ERR_UNSUPPORTED";
    case DP_ERR_ALIAS: return "DP_ERR_ALIAS";
    case DP_ERR_CUDA: return "DP_ERR_CUDA";
    case DP_ERR_TIMEOUT: return "DP_ERR_TIMEOUT";
  }
  return "DP_ERR_UNKNOWN";
}

int dp_version(void) { return 100; }  // 0.1.0

dp_status_t dp_reduce_scatter_dual(const void* const* bufs, int K, size_t N, dp_dtype_t in_dtype,
                                   float* const* out_f32, void* const* out_bf16, float scale,
                                   dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_reduce_scatter_dual");
  if (!bufs || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (!out_f32 && !out_bf16) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(in_dtype)) return DP_ERR_UNSUPPORTED;
  if (N % (size_t)K) return DP_ERR_INVALID_ARG;
  const size_t C = N / (size_t)K;
  Range rin[DP_MAX_K], rout[2 * DP_MAX_K];
  int nout = 0;
  bool vec = (C % 8) == 0;
  for (int r = 0; r < K; ++r) {
    if (!bufs[r]) return DP_ERR_INVALID_ARG;
    if (out_f32 && !out_f32[r]) return DP_ERR_INVALID_ARG;
    if (out_bf16 && !out_bf16[r]) return DP_ERR_INVALID_ARG;
    rin[r] = range_of(bufs[r], N * dtype_size(in_dtype));
    if (out_f32) rout[nout++] = range_of(out_f32[r], C * 4);
    if (out_bf16) rout[nout++] = range_of(out_bf16[r], C * 2);
    vec = vec && aligned16(bufs[r]) && (!out_f32 || aligned16(out_f32[r])) &&
          (!out_bf16 || aligned16(out_bf16[r]));
  }
  if (N == 0) return DP_OK;
  if (any_overlap(rout, nout, rin, K)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  dpl::RsArgs a{};
  for (int r = 0; r < K; ++r) {
    a.in[r] = bufs[r];
    a.out32[r] = out_f32 ? out_f32[r] : nullptr;
    a.out16[r] = out_bf16 ? static_cast<uint16_t*>(out_bf16[r]) : nullptr;
  }
  a.K = K;
  a.N = N;
  a.C = C;
  a.scale = scale;
  a.in_dtype = in_dtype;
  a.vec_ok = vec;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (vec && dph::collective_variant() == dph::kVariantBulkCopy)
    return from_cuda(dpl::launch_reduce_scatter_tma(a, dev, cs));
  return from_cuda(dpl::launch_reduce_scatter(a, dev, cs));
}

dp_status_t dp_reduce_scatter(const void* const* bufs, int K, size_t N, dp_dtype_t in_dtype,
                              void* const* out_shards, float scale, dp_dtype_t out_dtype,
                              dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_reduce_scatter");
  if (!out_shards) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(out_dtype)) return DP_ERR_UNSUPPORTED;
  if (out_dtype == DP_FP32)
    return dp_reduce_scatter_dual(bufs, K, N, in_dtype,
                                  reinterpret_cast<float* const*>(out_shards), nullptr, scale,
                                  stream);
  return dp_reduce_scatter_dual(bufs, K, N, in_dtype, nullptr, out_shards, scale, stream);
}

dp_status_t dp_all_gather(const void* const* shards, int K, size_t shard_elems, dp_dtype_t dtype,
                          void* const* out, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_all_gather");
  if (!shards || !out || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return DP_ERR_UNSUPPORTED;
  const size_t esz = dtype_size(dtype);
  Range rin[DP_MAX_K], rout[DP_MAX_K];
  bool vec = ((shard_elems * esz) % 16) == 0;
  for (int r = 0; r < K; ++r) {
    if (!shards[r] || !out[r]) return DP_ERR_INVALID_ARG;
    rin[r] = range_of(shards[r], shard_elems * esz);
    rout[r] = range_of(out[r], (size_t)K * shard_elems * esz);
    vec = vec && aligned16(shards[r]) && aligned16(out[r]);
  }
  if (shard_elems == 0) return DP_OK;
  if (any_overlap(rout, K, rin, K)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  dpl::AgArgs a{};
  for (int r = 0; r < K; ++r) {
    a.shards[r] = shards[r];
    a.out[r] = out[r];
  }
  a.K = K;
  a.C = shard_elems;
  a.esz = esz;
  a.vec_ok = vec;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (vec && use_bulk_copy()) return from_cuda(dpl::launch_all_gather_tma(a, dev, cs));
  return from_cuda(dpl::launch_all_gather(a, dev, cs));
}

dp_status_t dp_ring_allreduce(void* const* bufs, int K, size_t N, dp_dtype_t dtype, float scale,
                              dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_ring_allreduce");
  if (!bufs || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return DP_ERR_UNSUPPORTED;
  const size_t C = (N + (size_t)K - 1) / (size_t)K;
  Range rb[DP_MAX_K];
  bool vec = (C % 8) == 0;
  for (int r = 0; r < K; ++r) {
    if (!bufs[r]) return DP_ERR_INVALID_ARG;
    rb[r] = range_of(bufs[r], N * dtype_size(dtype));
    vec = vec && aligned16(bufs[r]);
  }
  if (N == 0) return DP_OK;
  if (any_overlap(rb, K, nullptr, 0)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  dpl::ArArgs a{};
  for (int r = 0; r < K; ++r) a.bufs[r] = bufs[r];
  a.K = K;
  a.N = N;
  a.C = C;
  a.scale = scale;
  a.dtype = dtype;
  a.vec_ok = vec;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (vec && all_reduce_bulk(N * dtype_size(dtype))) return from_cuda(dpl::launch_all_reduce_tma(a, dev, cs));
  return from_cuda(dpl::launch_all_reduce(a, dev, cs));
}

dp_status_t dp_grad_accumulate(float* acc, const void* grad, size_t N, dp_dtype_t grad_dtype,
                               int first, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_grad_accumulate");
  if (!acc) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(grad_dtype)) return DP_ERR_UNSUPPORTED;
  if (N == 0) return DP_OK;
  if (grad) {
    Range ra = range_of(acc, N * 4), rg = range_of(grad, N * dtype_size(grad_dtype));
    if (overlaps(ra, rg)) return DP_ERR_ALIAS;
  }
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  dpl::AccArgs a{};
  a.acc = acc;
  a.grad = grad;
  a.N = N;
  a.grad_dtype = grad_dtype;
  a.first = first != 0;
  a.vec_ok = aligned16(acc) && (!grad || aligned16(grad));
  return from_cuda(dpl::launch_accumulate(a, dev, reinterpret_cast<cudaStream_t>(stream)));
}

dp_status_t dp_odc_reduce_scatter(const void* const* grads, const int* m, int K, int Mmax,
                                  size_t N, dp_dtype_t grad_dtype, float* const* out_f32,
                                  void* const* out_bf16, float scale, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_odc_reduce_scatter");
  dpl::OdcArgs a;
  bool noop = false;
  dp_status_t st = dph::odc_prepare(grads, m, K, Mmax, N, grad_dtype, nullptr,
                                    DP_SETTLE_FIRST | DP_SETTLE_LAST, out_f32, out_bf16, scale,
                                    &a, &noop);
  if (st != DP_OK || noop) return st;
  return dph::odc_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dp_status_t dp_odc_settle_group(const void* const* grads, const int* m, int K, int Mmax,
                                size_t N, dp_dtype_t grad_dtype, float* const* owner_acc,
                                int phase, float* const* out_f32, void* const* out_bf16,
                                float scale, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_odc_settle_group");
  dpl::OdcArgs a;
  bool noop = false;
  dp_status_t st = dph::odc_prepare(grads, m, K, Mmax, N, grad_dtype, owner_acc, phase, out_f32,
                                    out_bf16, scale, &a, &noop);
  if (st != DP_OK || noop) return st;
  return dph::odc_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dp_status_t dp_allgather_matmul(const void* x_local, int M, int D, const void* const* w_shards,
                                int K, int F_shard, void* y, dp_dtype_t y_dtype,
                                void* workspace, size_t workspace_bytes, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_allgather_matmul");
  if (!x_local || !w_shards || !y || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (!workspace) workspace_bytes = 0;
  if (workspace_bytes && !aligned16(workspace)) return DP_ERR_UNSUPPORTED;
  if (M < 0 || D < 0 || F_shard < 0) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(y_dtype)) return DP_ERR_UNSUPPORTED;
  if ((D % 8) != 0 || (F_shard % 16) != 0) return DP_ERR_UNSUPPORTED;
  if (!aligned16(x_local) || !aligned16(y)) return DP_ERR_UNSUPPORTED;
  Range rin[DP_MAX_K + 1];
  for (int k = 0; k < K; ++k) {
    if (!w_shards[k]) return DP_ERR_INVALID_ARG;
    if (!aligned16(w_shards[k])) return DP_ERR_UNSUPPORTED;
    rin[k] = range_of(w_shards[k], (size_t)F_shard * (size_t)D * 2);
  }
  rin[K] = range_of(x_local, (size_t)M * (size_t)D * 2);
  const size_t F = (size_t)K * (size_t)F_shard;
  if (M == 0 || F == 0) return DP_OK;
  Range rw[2] = {range_of(y, (size_t)M * F * dtype_size(y_dtype)),
                 range_of(workspace, workspace_bytes)};
  if (any_overlap(rw, workspace_bytes ? 2 : 1, rin, K + 1)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 0) return from_cuda(cudaMemsetAsync(y, 0, (size_t)M * F * dtype_size(y_dtype), s));
  dpl::AgmmArgs a{};
  a.x = x_local;
  for (int k = 0; k < K; ++k) a.w[k] = w_shards[k];
  a.y = y;
  a.M = M;
  a.D = D;
  a.K = K;
  a.F_shard = F_shard;
  a.y_dtype = y_dtype;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  cudaError_t e = dpl::launch_allgather_matmul(a, dev, s);
  if (e == cudaErrorNotSupported) {
    cudaGetLastError();
    return DP_ERR_UNSUPPORTED;
  }
  return from_cuda(e);
}

}  // extern "C"

namespace {

dp_status_t matmul_reduce(const void* const* x_shards, const void* const* w_shards, int K, int M,
                          int D_shard, int F, void* const* y_out, dp_dtype_t y_dtype,
                          float scale, bool scatter, bool w_kn, void* workspace,
                          size_t workspace_bytes, dp_stream_t stream) {
  if (!x_shards || !w_shards || !y_out || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (!workspace) workspace_bytes = 0;
  if (workspace_bytes && !aligned16(workspace)) return DP_ERR_UNSUPPORTED;
  if (M < 0 || D_shard < 0 || F < 0) return DP_ERR_INVALID_ARG;
  if (scatter && (M % K) != 0) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(y_dtype)) return DP_ERR_UNSUPPORTED;
  if ((D_shard % 8) != 0 || (F % 16) != 0) return DP_ERR_UNSUPPORTED;
  if (w_kn && (F % 64) != 0) return DP_ERR_UNSUPPORTED;  // 64-column slabs of w_r
  const size_t ysz = dtype_size(y_dtype);
  const size_t out_rows = scatter ? (size_t)(M / K) : (size_t)M;
  Range rin[2 * DP_MAX_K], rout[DP_MAX_K + 1];
  for (int r = 0; r < K; ++r) {
    if (!x_shards[r] || !w_shards[r] || !y_out[r]) return DP_ERR_INVALID_ARG;
    if (!aligned16(x_shards[r]) || !aligned16(w_shards[r]) || !aligned16(y_out[r]))
      return DP_ERR_UNSUPPORTED;
    rin[2 * r] = range_of(x_shards[r], (size_t)M * (size_t)D_shard * 2);
    rin[2 * r + 1] = range_of(w_shards[r], (size_t)F * (size_t)D_shard * 2);
    rout[r] = range_of(y_out[r], out_rows * (size_t)F * ysz);
  }
  int nout = K;
  if (workspace_bytes) rout[nout++] = range_of(workspace, workspace_bytes);
  if (M == 0 || F == 0) return DP_OK;
  if (any_overlap(rout, nout, rin, 2 * K)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D_shard == 0) {
    for (int r = 0; r < K; ++r)
      if (cudaMemsetAsync(y_out[r], 0, out_rows * (size_t)F * ysz, s) != cudaSuccess)
        return DP_ERR_CUDA;
    return DP_OK;
  }
  dpl::MmrArgs a{};
  for (int r = 0; r < K; ++r) {
    a.x[r] = x_shards[r];
    a.w[r] = w_shards[r];
    a.y[r] = y_out[r];
  }
  a.M = M;
  a.D_shard = D_shard;
  a.F = F;
  a.K = K;
  a.scale = scale;
  a.y_dtype = y_dtype;
  a.scatter = scatter;
  a.w_kn = w_kn;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  cudaError_t e = dpl::launch_matmul_reduce(a, dev, s);
  if (e == cudaErrorNotSupported) {
    cudaGetLastError();
    return DP_ERR_UNSUPPORTED;
  }
  return from_cuda(e);
}

dp_status_t wgrad_reduce_scatter(const void* const* dy, const void* const* x, int K, int T, int F,
                                 int D, void* const* dw_shards, dp_dtype_t dw_dtype, float scale,
                                 void* workspace, size_t workspace_bytes, dp_stream_t stream) {
  if (!dy || !x || !dw_shards || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (T < 0 || F < 0 || D < 0) return DP_ERR_INVALID_ARG;
  if ((F % K) != 0) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(dw_dtype)) return DP_ERR_UNSUPPORTED;
  if ((F % 64) != 0 || (D % 64) != 0) return DP_ERR_UNSUPPORTED;
  const size_t ysz = dtype_size(dw_dtype);
  const size_t out_rows = (size_t)(F / K);
  if (!workspace) workspace_bytes = 0;
  if (workspace_bytes && !aligned16(workspace)) return DP_ERR_UNSUPPORTED;
  Range rin[2 * DP_MAX_K], rout[DP_MAX_K + 1];
  for (int r = 0; r < K; ++r) {
    if (!dy[r] || !x[r] || !dw_shards[r]) return DP_ERR_INVALID_ARG;
    if (!aligned16(dy[r]) || !aligned16(x[r]) || !aligned16(dw_shards[r]))
      return DP_ERR_UNSUPPORTED;
    rin[2 * r] = range_of(dy[r], (size_t)T * (size_t)F * 2);
    rin[2 * r + 1] = range_of(x[r], (size_t)T * (size_t)D * 2);
    rout[r] = range_of(dw_shards[r], out_rows * (size_t)D * ysz);
  }
  int nout = K;
  if (workspace_bytes) rout[nout++] = range_of(workspace, workspace_bytes);
  if (F == 0 || D == 0) return DP_OK;
  if (any_overlap(rout, nout, rin, 2 * K)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {  // no tokens: the gradient is zero
    for (int r = 0; r < K; ++r)
      if (cudaMemsetAsync(dw_shards[r], 0, out_rows * (size_t)D * ysz, s) != cudaSuccess)
        return DP_ERR_CUDA;
    return DP_OK;
  }
  dpl::WgradArgs a{};
  for (int r = 0; r < K; ++r) {
    a.dy[r] = dy[r];
    a.x[r] = x[r];
    a.y[r] = dw_shards[r];
  }
  a.T = T;
  a.F = F;
  a.D = D;
  a.K = K;
  a.scale = scale;
  a.y_dtype = dw_dtype;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  cudaError_t e = dpl::launch_wgrad_reduce_scatter(a, dev, s);
  if (e == cudaErrorNotSupported) {
    cudaGetLastError();
    return DP_ERR_UNSUPPORTED;
  }
  return from_cuda(e);
}

}  // namespace

extern "C" {

dp_status_t dp_wgrad_reduce_scatter(const void* const* dy, const void* const* x, int K, int T,
                                    int F, int D, void* const* dw_shards, dp_dtype_t dw_dtype,
                                    float scale, void* workspace, size_t workspace_bytes,
                                    dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_wgrad_reduce_scatter");
  return wgrad_reduce_scatter(dy, x, K, T, F, D, dw_shards, dw_dtype, scale, workspace,
                              workspace_bytes, stream);
}

dp_status_t dp_wgrad_workspace_size(int K, int T, int F, int D, size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  *bytes = 0;
  if (K < 1 || K > DP_MAX_K || T < 0 || F < 0 || D < 0) return DP_ERR_INVALID_ARG;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  *bytes = dpl::wgrad_workspace_bytes(K, T, F, D, dev);
  return DP_OK;
}

dp_status_t dp_matmul_allreduce(const void* const* x_shards, const void* const* w_shards, int K,
                                int M, int D_shard, int F, void* const* y_out,
                                dp_dtype_t y_dtype, float scale, void* workspace,
                                size_t workspace_bytes, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_matmul_allreduce");
  return matmul_reduce(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale, false, false,
                       workspace, workspace_bytes, stream);
}

dp_status_t dp_matmul_allreduce_xw(const void* const* x_shards, const void* const* w_shards,
                                   int K, int M, int D_shard, int F, void* const* y_out,
                                   dp_dtype_t y_dtype, float scale, void* workspace,
                                   size_t workspace_bytes, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_matmul_allreduce_xw");
  return matmul_reduce(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale, false, true,
                       workspace, workspace_bytes, stream);
}

dp_status_t dp_matmul_reduce_scatter_xw(const void* const* x_shards,
                                        const void* const* w_shards, int K, int M, int D_shard,
                                        int F, void* const* y_out, dp_dtype_t y_dtype,
                                        float scale, void* workspace, size_t workspace_bytes,
                                        dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_matmul_reduce_scatter_xw");
  return matmul_reduce(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale, true, true,
                       workspace, workspace_bytes, stream);
}

dp_status_t dp_matmul_reduce_scatter(const void* const* x_shards, const void* const* w_shards,
                                     int K, int M, int D_shard, int F, void* const* y_out,
                                     dp_dtype_t y_dtype, float scale, void* workspace,
                                     size_t workspace_bytes, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_matmul_reduce_scatter");
  return matmul_reduce(x_shards, w_shards, K, M, D_shard, F, y_out, y_dtype, scale, true, false,
                       workspace, workspace_bytes, stream);
}

dp_status_t dp_allgather_matmul_workspace_size(int M, int D, int K, int F_shard, size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  *bytes = 0;
  if (K < 1 || K > DP_MAX_K || M < 0 || D < 0 || F_shard < 0) return DP_ERR_INVALID_ARG;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  *bytes = dpl::allgather_matmul_workspace_bytes(M, D, K, F_shard, dev);
  return DP_OK;
}

dp_status_t dp_matmul_workspace_size(int K, int M, int D_shard, int F, size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  *bytes = 0;
  if (K < 1 || K > DP_MAX_K || M < 0 || D_shard < 0 || F < 0) return DP_ERR_INVALID_ARG;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  *bytes = dpl::matmul_reduce_workspace_bytes(K, M, D_shard, F, false, dev);
  return DP_OK;
}

dp_status_t dp_matmul_xw_workspace_size(int K, int M, int D_shard, int F, size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  *bytes = 0;
  if (K < 1 || K > DP_MAX_K || M < 0 || D_shard < 0 || F < 0) return DP_ERR_INVALID_ARG;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  *bytes = dpl::matmul_reduce_workspace_bytes(K, M, D_shard, F, true, dev);
  return DP_OK;
}

}  // extern "C"

extern "C" {

dp_status_t dp_get_device_error(dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_get_device_error");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return DP_ERR_CUDA;
  }
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  unsigned w = 0;
  if (cudaMemcpy(&w, dev.err_word, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return DP_ERR_CUDA;
  }
  if (w == 0) return DP_OK;
  const unsigned zero = 0;
  if (cudaMemcpy(dev.err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return DP_ERR_CUDA;
  }
  return (w & dpk::kErrTimeout) ? DP_ERR_TIMEOUT : DP_ERR_CUDA;
}

dp_status_t dp_set_collective_variant(int variant) {
  if (variant < 0 || variant > 2) return DP_ERR_INVALID_ARG;
  dph::set_collective_variant(variant);
  return DP_OK;
}

int dp_get_collective_variant(void) { return dph::collective_variant(); }

dp_status_t dp_set_cta_limits(int gemm_ctas, int stream_ctas) {
  if (gemm_ctas < 0 || stream_ctas < 0) return DP_ERR_INVALID_ARG;
  dph::set_cta_limits(gemm_ctas, stream_ctas);
  return DP_OK;
}

dp_status_t dp_get_cta_limits(int* gemm_ctas, int* stream_ctas) {
  if (gemm_ctas) *gemm_ctas = dph::gemm_cta_limit();
  if (stream_ctas) *stream_ctas = dph::stream_cta_limit();
  return DP_OK;
}

}  // extern "C"

namespace {

// Internal streams of the copy-engine all-gather, created once per device.
// Copies issued on one stream run one after another on one DMA engine.  The
// copies are issued shard by shard, destination r on stream r % streams, so
// that the engines read the same shard at the same time and all but the
// first read of it hit L2.  Measured on GB300 from a CUDA graph, 8 x 8
// copies of 16 MiB (32 MiB): destination by destination on 1 / 2 / 4 / 8
// streams 0.437 / 0.319 / 0.319 / 0.319 ms (0.748 / 0.629 / 0.628 / 0.629),
// shard by shard 0.310 / 0.211 / 0.196 / 0.214 ms (0.561 / 0.443 / 0.442 /
// 0.443).
constexpr int kCopyStreams = 4;
struct CopyStreams {
  cudaStream_t s[kCopyStreams];
  cudaEvent_t fork;
  cudaEvent_t join[kCopyStreams];
};
std::mutex g_ce_mutex;  // guards the table and orders the issue of each call
CopyStreams g_ce[64];
bool g_ce_ready[64] = {};

// The current device's copy streams (device `dev` must be current); nullptr
// if they cannot be created.  Call with g_ce_mutex held.
CopyStreams* copy_streams(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  if (g_ce_ready[dev]) return &g_ce[dev];
  CopyStreams& cs = g_ce[dev];
  bool ok = cudaEventCreateWithFlags(&cs.fork, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kCopyStreams; ++i)
    ok = cudaStreamCreateWithFlags(&cs.s[i], cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&cs.join[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return nullptr;
  }
  g_ce_ready[dev] = true;
  return &cs;
}

}  // namespace

extern "C" {

dp_status_t dp_all_gather_copy_engine(const void* const* shards, int K, size_t shard_elems,
                                      dp_dtype_t dtype, void* const* out, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_all_gather_copy_engine");
  if (!shards || !out || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return DP_ERR_UNSUPPORTED;
  const size_t esz = dtype_size(dtype);
  const size_t bytes = shard_elems * esz;
  Range rin[DP_MAX_K], rout[DP_MAX_K];
  for (int r = 0; r < K; ++r) {
    if (!shards[r] || !out[r]) return DP_ERR_INVALID_ARG;
    rin[r] = range_of(shards[r], bytes);
    rout[r] = range_of(out[r], (size_t)K * bytes);
  }
  if (bytes == 0) return DP_OK;
  if (any_overlap(rout, K, rin, K)) return DP_ERR_ALIAS;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // One device-to-device copy per (destination rank, shard): the DMA engines
  // move the data while the SMs stay free for other work.  The copies are
  // spread over the device's internal copy streams, forked from and joined
  // back to `s` through events, so several engines run at once, each on a
  // different destination of the same shard.
  std::lock_guard<std::mutex> lock(g_ce_mutex);
  CopyStreams* cs = copy_streams(dev.device);
  if (!cs) return DP_ERR_CUDA;
  bool ok = cudaEventRecord(cs->fork, s) == cudaSuccess;
  for (int i = 0; ok && i < kCopyStreams; ++i)
    ok = cudaStreamWaitEvent(cs->s[i], cs->fork, 0) == cudaSuccess;
  for (int c = 0; ok && c < K; ++c)
    for (int r = 0; ok && r < K; ++r)
      ok = cudaMemcpyAsync(static_cast<unsigned char*>(out[r]) + (size_t)c * bytes, shards[c],
                           bytes, cudaMemcpyDeviceToDevice, cs->s[r % kCopyStreams]) ==
           cudaSuccess;
  for (int i = 0; i < kCopyStreams; ++i) {  // join even after a failure
    const bool rec = cudaEventRecord(cs->join[i], cs->s[i]) == cudaSuccess;
    ok = rec && cudaStreamWaitEvent(s, cs->join[i], 0) == cudaSuccess && ok;
  }
  if (!ok) {
    cudaGetLastError();
    return DP_ERR_CUDA;
  }
  return DP_OK;
}

dp_status_t dp_selftest_bounded_wait(uint32_t timeout_us, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_selftest_bounded_wait");
  if (timeout_us < 1 || timeout_us > 2000000u) return DP_ERR_INVALID_ARG;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  return from_cuda(
      dpl::launch_selftest_wait(timeout_us, dev, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
