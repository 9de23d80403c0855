// dp_pipe.cu -- the cross-iteration settle pipeline ("Using ODC to
// Accelerate AMD SFT Training", section "Discussion: Settle Does Not Yet
// Overlap with Backward": a separate stream and events let the previous
// microbatch group's settle run beside this group's backward compute, with
// one join per minibatch).
//
// A pipe owns one non-blocking stream and two events on one device.  A push
// records the point in the caller's stream where a group's gradients are
// complete, makes the pipe's stream wait for that point and enqueues the
// group's settle (dp_odc_settle_group's kernel) there; the caller's stream
// is not held back.  A wait records the pipe's progress and makes the
// caller's stream wait for it.  Host code only: every step of the settle
// runs in the fused settle kernel.

#include "dp_launch.h"

#include <mutex>
#include <new>

struct dp_settle_pipe {
  int device = -1;
  int cta_limit = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t ready = nullptr;  // a group's gradients are complete (caller's stream)
  cudaEvent_t done = nullptr;   // every settle pushed so far (pipe's stream)
  std::mutex mu;
};

namespace {

dp_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DP_OK;
  cudaGetLastError();
  return DP_ERR_CUDA;
}

bool on_pipe_device(const dp_settle_pipe* p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return dev == p->device;
}

void release(dp_settle_pipe* p) {
  if (p->done) cudaEventDestroy(p->done);
  if (p->ready) cudaEventDestroy(p->ready);
  if (p->side) cudaStreamDestroy(p->side);
  delete p;
}

}  // namespace

extern "C" {

dp_status_t dp_settle_pipe_create(int cta_limit, dp_settle_pipe_t** out) {
  if (!out || cta_limit < 0) return DP_ERR_INVALID_ARG;
  *out = nullptr;
  dp_settle_pipe* p = new (std::nothrow) dp_settle_pipe;
  if (!p) return DP_ERR_CUDA;
  p->cta_limit = cta_limit;
  dp_status_t st = cuda_status(cudaGetDevice(&p->device));
  if (st == DP_OK) st = cuda_status(cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking));
  if (st == DP_OK)
    st = cuda_status(cudaEventCreateWithFlags(&p->ready, cudaEventDisableTiming));
  if (st == DP_OK) st = cuda_status(cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming));
  if (st != DP_OK) {
    release(p);
    return st;
  }
  *out = p;
  return DP_OK;
}

dp_status_t dp_settle_pipe_push(dp_settle_pipe_t* p, const void* const* grads, const int* m,
                                int K, int Mmax, size_t N, dp_dtype_t grad_dtype,
                                float* const* owner_acc, int phase, float* const* out_f32,
                                void* const* out_bf16, float scale, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_settle_pipe_push");
  if (!p) return DP_ERR_INVALID_ARG;
  dpl::OdcArgs a;
  bool noop = false;
  dp_status_t st = dph::odc_prepare(grads, m, K, Mmax, N, grad_dtype, owner_acc, phase, out_f32,
                                    out_bf16, scale, &a, &noop);
  if (st != DP_OK || noop) return st;
  a.cta_limit = p->cta_limit;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!on_pipe_device(p)) return DP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = cuda_status(cudaEventRecord(p->ready, s));
  if (st == DP_OK) st = cuda_status(cudaStreamWaitEvent(p->side, p->ready, 0));
  if (st == DP_OK) st = dph::odc_launch(a, p->side);
  return st;
}

dp_status_t dp_settle_pipe_wait(dp_settle_pipe_t* p, dp_stream_t stream) {
  if (!p) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!on_pipe_device(p)) return DP_ERR_INVALID_ARG;
  dp_status_t st = cuda_status(cudaEventRecord(p->done, p->side));
  if (st == DP_OK)
    st = cuda_status(cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), p->done, 0));
  return st;
}

dp_status_t dp_settle_pipe_destroy(dp_settle_pipe_t* p) {
  if (!p) return DP_ERR_INVALID_ARG;
  dp_status_t st = DP_OK;
  {
    std::lock_guard<std::mutex> lock(p->mu);
    int prev = -1;
    if (cudaGetDevice(&prev) == cudaSuccess && prev != p->device) cudaSetDevice(p->device);
    st = cuda_status(cudaStreamSynchronize(p->side));
    if (prev >= 0 && prev != p->device) cudaSetDevice(prev);
  }
  release(p);
  return st;
}

}  // extern "C"
