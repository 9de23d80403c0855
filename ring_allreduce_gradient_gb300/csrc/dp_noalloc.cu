// dp_noalloc.cu -- the weight-gradient reduce-scatter for callers that cannot
// allocate device memory.
//
// dp_wgrad_reduce_scatter runs fastest with a scratch workspace that the
// caller allocates.  Some callers cannot do that: code that runs under a
// framework whose memory pool owns the whole GPU and forbids allocations
// behind its back, code that cannot afford the implicit device-wide
// synchronisation of cudaMalloc / cudaFree in the middle of a training step,
// and code with a fixed device-memory budget settled at start-up.  For them,
// dp_wgrad_reduce_scatter_noalloc takes its scratch from the array below,
// which the CUDA runtime places in device memory when it loads this library
// onto a GPU and which stays there until the process exits.  The call itself
// allocates nothing.

#include "dp_launch.h"

#include <mutex>

namespace {

constexpr size_t kScratchBytes = DP_WGRAD_NOALLOC_MAX_BYTES;

// Scratch shared by every call on a device.  Its name, used in host code, is
// only a host-side stand-in: the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_wgrad_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up on
// the first call per device, with that device current).
dp_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DP_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return DP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return DP_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DP_OK;
}

}  // namespace

extern "C" {

dp_status_t dp_wgrad_reduce_scatter_noalloc(const void* const* dy, const void* const* x, int K,
                                            int T, int F, int D, void* const* dw_shards,
                                            dp_dtype_t dw_dtype, float scale,
                                            dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_wgrad_reduce_scatter_noalloc");
  size_t need = 0;
  dp_status_t st = dp_wgrad_workspace_size(K, T, F, D, &need);
  if (st != DP_OK) return st;
  if (need > kScratchBytes) return DP_ERR_UNSUPPORTED;  // beyond the built-in scratch
  void* scratch = nullptr;
  if (need) {
    st = scratch_address(&scratch);
    if (st != DP_OK) return st;
    // The array keeps whatever the previous call left in it, and nothing
    // needs clearing: every call tags its hand-off flags with a 64-bit value
    // of its own, a stale flag never carries it, and partial sums are only
    // read after their flag does.
  }
  return dp_wgrad_reduce_scatter(dy, x, K, T, F, D, dw_shards, dw_dtype, scale, scratch, need,
                                 stream);
}

}  // extern "C"
