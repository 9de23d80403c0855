// dp_common.cuh -- device helpers and host plumbing shared by the kernels of
// libdp_gb300 (product code only; nothing here is used by the oracle).  The
// launchers' argument structs live in dp_launch.h.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/dp.h"

namespace dpk {

constexpr int kMaxK = DP_MAX_K;
constexpr int kMaxMb = DP_MAX_MICROBATCHES;

// Bits of the device error word.
constexpr unsigned kErrTimeout = 1u;

// ---------------------------------------------------------------------------
// 128-bit global memory access.  Inputs are read once, so they bypass L1 and
// carry an L2 128-byte prefetch hint (measured on GB300 against 256 bytes and
// no size hint, the K=8 bf16 reduce-scatter streams 6.54 / 6.49 / 6.53 TB/s);
// outputs use the streaming store.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Plain (coherent) 128-bit load, for buffers the same kernel also writes.
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32.  Widening is exact (bf16 is the top half of a binary32).
// Narrowing uses the hardware's round-to-nearest-even conversion.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  // cvt packs its first source into the upper half.
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t bf16_rn(float f) {
  return (uint16_t)(pack_bf16x2_rn(f, 0.0f) & 0xffffu);
}

// Eight consecutive elements of type T, widened to fp32.
template <typename T>
struct Vec8;

template <>
struct Vec8<float> {
  static constexpr int kLoads = 2;  // two 16-byte loads
  __device__ __forceinline__ static void load(const float* p, uint4 (&raw)[2]) {
    raw[0] = ld_stream_v4(p);
    raw[1] = ld_stream_v4(p + 4);
  }
  __device__ __forceinline__ static void load_rw(const float* p, uint4 (&raw)[2]) {
    raw[0] = ld_v4(p);
    raw[1] = ld_v4(p + 4);
  }
  __device__ __forceinline__ static void widen(const uint4 (&raw)[2], float (&v)[8]) {
    v[0] = __uint_as_float(raw[0].x); v[1] = __uint_as_float(raw[0].y);
    v[2] = __uint_as_float(raw[0].z); v[3] = __uint_as_float(raw[0].w);
    v[4] = __uint_as_float(raw[1].x); v[5] = __uint_as_float(raw[1].y);
    v[6] = __uint_as_float(raw[1].z); v[7] = __uint_as_float(raw[1].w);
  }
};

template <>
struct Vec8<uint16_t> {
  static constexpr int kLoads = 1;  // one 16-byte load
  __device__ __forceinline__ static void load(const uint16_t* p, uint4 (&raw)[1]) {
    raw[0] = ld_stream_v4(p);
  }
  __device__ __forceinline__ static void load_rw(const uint16_t* p, uint4 (&raw)[1]) {
    raw[0] = ld_v4(p);
  }
  __device__ __forceinline__ static void widen(const uint4 (&raw)[1], float (&v)[8]) {
    v[0] = bf16lo(raw[0].x); v[1] = bf16hi(raw[0].x);
    v[2] = bf16lo(raw[0].y); v[3] = bf16hi(raw[0].y);
    v[4] = bf16lo(raw[0].z); v[5] = bf16hi(raw[0].z);
    v[6] = bf16lo(raw[0].w); v[7] = bf16hi(raw[0].w);
  }
};

__device__ __forceinline__ float widen_scalar(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float widen_scalar(const uint16_t* p, size_t i) {
  return __uint_as_float((uint32_t)p[i] << 16);
}

// Store eight fp32 values as fp32 (32 bytes) or bf16 (16 bytes).
__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8]) {
  st_stream_v4(p, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                             __float_as_uint(v[2]), __float_as_uint(v[3])));
  st_stream_v4(p + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                 __float_as_uint(v[6]), __float_as_uint(v[7])));
}
__device__ __forceinline__ void store8_bf16(uint16_t* p, const float (&v)[8]) {
  st_stream_v4(p, make_uint4(pack_bf16x2_rn(v[0], v[1]), pack_bf16x2_rn(v[2], v[3]),
                             pack_bf16x2_rn(v[4], v[5]), pack_bf16x2_rn(v[6], v[7])));
}

// ---------------------------------------------------------------------------
// Bounded waits.  Every spin on an mbarrier gives up after a deadline taken
// from the global nanosecond timer, records kErrTimeout in the device error
// word and reports failure to the caller, which then unwinds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed, or until
// `timeout_ns` has passed.  Returns false (and flags the error word) on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned* err_word, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u && globaltimer_ns() - t0 > timeout_ns) {
      atomicOr(err_word, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

}  // namespace dpk

// ---------------------------------------------------------------------------
// Host-side launch plumbing (implemented in dp_api.cu).
// ---------------------------------------------------------------------------
namespace dph {

// An NVTX range around one entry point, visible to profilers that attach
// (Nsight Systems / Compute); a no-op otherwise.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
  unsigned* err_word = nullptr;  // device address of the error word
};

// Info for the current device (cached per device).  Returns false if there
// is no usable device.
bool current_device(DeviceInfo* out);

// Prepares `kernel` for launches with `smem` bytes of dynamic shared memory
// on device `device` (the attribute is set once per kernel and device) and
// returns its resident CTAs per SM with `threads` threads; 0 on failure.
int prepare_kernel(const void* kernel, int threads, size_t smem, int device);

// Process-wide CTA limits set by dp_set_cta_limits (0 = no limit).
int gemm_cta_limit();
int stream_cta_limit();
void set_cta_limits(int gemm_ctas, int stream_ctas);

// Implementation variant of the all-reduce / all-gather (dp_set_collective_variant).
enum { kVariantAuto = 0, kVariantRegisters = 1, kVariantBulkCopy = 2 };
int collective_variant();
void set_collective_variant(int v);

}  // namespace dph

