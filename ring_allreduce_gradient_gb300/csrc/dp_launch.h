// dp_launch.h -- the launchers' argument structs and declarations: the
// host-side interface between the C entry points (dp_api.cu and the Reducer)
// and the kernel translation units.  Host code only.
#pragma once

#include "dp_common.cuh"

// Launchers (host functions defined in the kernel translation units).  They
// assume validated arguments and return the launch status.
namespace dpl {

struct RsArgs {
  const void* in[DP_MAX_K];
  float* out32[DP_MAX_K];
  uint16_t* out16[DP_MAX_K];
  int K;
  size_t N;
  size_t C;
  float scale;
  dp_dtype_t in_dtype;
  bool vec_ok;
};
cudaError_t launch_reduce_scatter(const RsArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_reduce_scatter_tma(const RsArgs& a, const dph::DeviceInfo& dev,
                                      cudaStream_t s);

struct AgArgs {
  const void* shards[DP_MAX_K];
  void* out[DP_MAX_K];
  int K;
  size_t C;  // elements per shard
  size_t esz;
  bool vec_ok;
};
cudaError_t launch_all_gather(const AgArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_all_gather_tma(const AgArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);

struct ArArgs {
  void* bufs[DP_MAX_K];
  int K;
  size_t N;
  size_t C;
  float scale;
  dp_dtype_t dtype;
  bool vec_ok;
};
cudaError_t launch_all_reduce(const ArArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_all_reduce_tma(const ArArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);

struct AccArgs {
  float* acc;
  const void* grad;
  size_t N;
  dp_dtype_t grad_dtype;
  bool first;
  bool vec_ok;
};
cudaError_t launch_accumulate(const AccArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);

struct OdcArgs {
  const void* grads[DP_MAX_K][DP_MAX_MICROBATCHES];
  int m[DP_MAX_K];
  float* out32[DP_MAX_K];
  uint16_t* out16[DP_MAX_K];
  float* carry[DP_MAX_K];  // owner accumulators of a pipelined settle
  int phase;               // DP_SETTLE_FIRST | DP_SETTLE_LAST bits (both: one settle)
  int cta_limit;           // > 0: grid cap for this launch (else the process-wide one)
  int K;
  size_t N;
  size_t C;
  float scale;
  dp_dtype_t grad_dtype;
  bool vec_ok;
};
cudaError_t launch_odc_reduce_scatter(const OdcArgs& a, const dph::DeviceInfo& dev,
                                      cudaStream_t s);
}  // namespace dpl

namespace dph {
// Argument checks of the variable-length settle calls (dp_api.cu): fills
// *a, or returns the error before anything is enqueued; *noop for N == 0.
dp_status_t odc_prepare(const void* const* grads, const int* m, int K, int Mmax, size_t N,
                        dp_dtype_t grad_dtype, float* const* owner_acc, int phase,
                        float* const* out_f32, void* const* out_bf16, float scale,
                        dpl::OdcArgs* a, bool* noop);
// Launch a prepared settle on the current device.
dp_status_t odc_launch(const dpl::OdcArgs& a, cudaStream_t s);
}  // namespace dph

namespace dpl {

struct AgmmArgs {
  const void* x;
  const void* w[DP_MAX_K];
  void* y;
  int M, D, K, F_shard;
  dp_dtype_t y_dtype;
  void* workspace;         // optional (nullptr): the chained split of the last round
  size_t workspace_bytes;
};
// Returns cudaErrorNotSupported for a device/shape the tensor-core path can't take.
cudaError_t launch_allgather_matmul(const AgmmArgs& a, const dph::DeviceInfo& dev,
                                    cudaStream_t s);
// Workspace bytes with which the gather GEMM splits its last round on `dev`
// under the current CTA limit (0: no split for this shape).
size_t allgather_matmul_workspace_bytes(int M, int D, int K, int F_shard,
                                        const dph::DeviceInfo& dev);

struct MmrArgs {
  const void* x[DP_MAX_K];  // rank r: x_r [M, D_shard] bf16
  const void* w[DP_MAX_K];  // rank r: w_r [F, D_shard] bf16
  void* y[DP_MAX_K];
  int M, D_shard, F, K;
  float scale;
  dp_dtype_t y_dtype;
  bool scatter;  // true: row shards (reduce-scatter); false: every rank (all-reduce)
  bool w_kn;     // w_r given [D_shard, F] row-major (the x . w orientation)
  void* workspace;  // optional (nullptr): the chained split of the last round
  size_t workspace_bytes;
};
cudaError_t launch_matmul_reduce(const MmrArgs& a, const dph::DeviceInfo& dev, cudaStream_t s);
// The same for the tensor-parallel GEMMs (all-reduce and reduce-scatter forms
// share their tiling).
size_t matmul_reduce_workspace_bytes(int K, int M, int D_shard, int F, bool w_kn,
                                     const dph::DeviceInfo& dev);

struct WgradArgs {
  const void* dy[DP_MAX_K];  // rank r: dY_r [T, F] bf16 (output gradients, tokens x features)
  const void* x[DP_MAX_K];   // rank r: X_r [T, D] bf16 (layer inputs)
  void* y[DP_MAX_K];         // shard c: rows [c*F/K, (c+1)*F/K) of dW [F, D]
  int T, F, D, K;
  float scale;
  dp_dtype_t y_dtype;
  void* workspace;         // optional (nullptr): the chained split of the last round
  size_t workspace_bytes;
};
cudaError_t launch_wgrad_reduce_scatter(const WgradArgs& a, const dph::DeviceInfo& dev,
                                        cudaStream_t s);
// Workspace bytes with which the weight gradient splits its last round on
// `dev` under the current CTA limit (0: no split for this shape).
size_t wgrad_workspace_bytes(int K, int T, int F, int D, const dph::DeviceInfo& dev);

struct BucketArgs {
  void* const* ptrs;      // n*K device pointers, tensor-major: ptrs[t*K + r]
  const size_t* numels;   // n element counts
  int n, K;
  float scale;
  dp_dtype_t dtype;
};
cudaError_t launch_bucket_allreduce(const BucketArgs& a, const dph::DeviceInfo& dev,
                                    cudaStream_t s);
cudaError_t launch_bucket_allreduce_tma(const BucketArgs& a, const dph::DeviceInfo& dev,
                                        cudaStream_t s);

cudaError_t launch_selftest_wait(uint32_t timeout_us, const dph::DeviceInfo& dev, cudaStream_t s);

}  // namespace dpl
