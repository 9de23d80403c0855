// dp_odc.cu -- microbatch accumulation and the variable-length settle.
//
// "Using ODC to Accelerate AMD SFT Training", sections "From Per-iteration to
// Per-minibatch Synchronization" and "odc_pad vs odc_nopad": each rank runs
// its own number of microbatches, accumulating their gradients into an fp32
// accumulator, and the accumulators are reduce-scattered once per minibatch.
// The accumulate kernel is the two-phase path (one launch per microbatch,
// then the ring reduce-scatter of the accumulators); the fused kernel reads
// every rank's microbatch gradients at an element once and settles in the
// same pass, with the same rounding as the two-phase path: microbatches
// ascending into a +0-seeded fp32 accumulator per rank, then the ring fold of
// the accumulators (x_{c+1} + ... + x_c) for chunk c.

#include "dp_stream_common.cuh"

namespace {

// ---------------------------------------------------------------------------
// Microbatch accumulation: acc = (first ? +0 : acc) + widen(g); g == NULL is
// a padding bucket (+0), which still costs the accumulator's read and write.
// ---------------------------------------------------------------------------
struct AccParams {
  float* acc;
  const void* grad;
  size_t N;
  size_t units;
};

template <typename Tg, bool FIRST, bool HAS_G>
__global__ void __launch_bounds__(kThreads) acc_vec_kernel(const __grid_constant__ AccParams p) {
  // Launched with programmatic stream serialization (a step accumulates
  // microbatch after microbatch): wait for the previous kernel of the stream
  // to complete and its writes to be visible, then let the next launch's
  // grid start scheduling.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const Tg* g = static_cast<const Tg*>(p.grad);
  const size_t T = (size_t)gridDim.x * kThreads;
  for (size_t u = (size_t)blockIdx.x * kThreads + threadIdx.x; u < p.units; u += T) {
    float base[8];
    if (FIRST) {
#pragma unroll
      for (int e = 0; e < 8; ++e) base[e] = 0.0f;
    } else {
      uint4 ra[2];
      Vec8<float>::load_rw(p.acc + u * 8, ra);
      Vec8<float>::widen(ra, base);
    }
    float gv[8];
    if (HAS_G) {
      uint4 rg[Vec8<Tg>::kLoads];
      Vec8<Tg>::load(g + u * 8, rg);
      Vec8<Tg>::widen(rg, gv);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) gv[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) base[e] = __fadd_rn(base[e], gv[e]);
    store8_f32(p.acc + u * 8, base);
  }
  // tail (N % 8 elements)
  if (blockIdx.x == 0) {
    for (size_t i = p.units * 8 + threadIdx.x; i < p.N; i += kThreads) {
      const float b = FIRST ? 0.0f : p.acc[i];
      const float gv = HAS_G ? widen_scalar(g, i) : 0.0f;
      p.acc[i] = __fadd_rn(b, gv);
    }
  }
}

template <typename Tg>
__global__ void __launch_bounds__(kThreads) acc_scalar_kernel(const __grid_constant__ AccParams p,
                                                              int first) {
  const Tg* g = static_cast<const Tg*>(p.grad);
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < p.N;
       i += (size_t)gridDim.x * kThreads) {
    const float b = first ? 0.0f : p.acc[i];
    const float gv = g ? widen_scalar(g, i) : 0.0f;
    p.acc[i] = __fadd_rn(b, gv);
  }
}

// ---------------------------------------------------------------------------
// Variable-length step, accumulate + settle in one pass.  For each element of
// chunk c: every rank's microbatch sum (+0) + g_0 + ... + g_{m-1} in fp32,
// then the ring fold of those K sums from rank c+1, the average and the
// casts.  Bit-identical to accumulating into K fp32 buffers and then running
// the reduce-scatter on them, without the accumulators' memory traffic.
// Padding buckets (NULL) add +0, which never changes a +0-seeded sum's bits,
// so their loads are skipped.
// ---------------------------------------------------------------------------
struct OdcParams {
  const void* grads[kMaxK][kMaxMb];
  int m[kMaxK];
  // The same gradients as one list for the vector kernel: the non-null ones,
  // rank by rank, microbatches ascending; first[i] marks the first of its
  // rank and pos[r] is where rank r's gradients start (for an empty rank,
  // where they would).  Padding buckets (null) are left out: they add +0.
  const void* items[kMaxK * kMaxMb];
  unsigned char first[kMaxK * kMaxMb];
  int pos[kMaxK];
  int n_items;
  float* out32[kMaxK];
  uint16_t* out16[kMaxK];
  // Owner accumulators of a pipelined settle (chunk c's fp32 running sum,
  // C elements each) and what this launch does with them (kSettle*).
  float* carry[kMaxK];
  int mode;
  int K;
  size_t C;
  size_t units;
  float scale;
};

// What a launch does with the settled chunk S (the ring fold of this
// launch's per-rank microbatch sums): the whole minibatch in one launch
// writes cast(S * scale); the first group of a pipelined settle stores S in
// the owner's accumulator (+0 + S), a middle group adds S to it, the last
// group writes cast((acc + S) * scale).
constexpr int kSettleWhole = 0, kSettleFirst = 1, kSettleMiddle = 2, kSettleLast = 3;

template <typename Tg, bool W32, bool W16, int MODE>
__global__ void __launch_bounds__(kThreads) odc_vec_kernel(const __grid_constant__ OdcParams p) {
  // Launched with programmatic stream serialization (a step settles one layer
  // after another): wait for the previous kernel of the stream to complete
  // and its writes to be visible before touching memory, then let the next
  // layer's grid start scheduling (32 layers: 6.77 -> 6.70 ms per step).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Loads are issued B at a time across the whole ring-ordered list of
  // gradients (8 in flight per thread whatever the microbatch counts, not
  // one rank's few at a time; measured on GB300 with microbatches [6, 7, 1,
  // 7, 4, 5, 6, 3]: 6.63 TB/s against 6.41 per rank; 16 at a time costs a
  // CTA per SM and measured 4.87); the arithmetic is the per-rank order: microbatches ascending
  // into a +0-seeded accumulator, then the ranks' accumulators folded in
  // ring order (c+1, ..., c).  The running total starts at +0 too, which is
  // bit-neutral because no accumulator is ever -0.
  constexpr int L = Vec8<Tg>::kLoads;
  constexpr int B = 8 / L;
  const int c = blockIdx.y;
  const int K = p.K;
  const int n = p.n_items;
  const int s0 = p.pos[c + 1 < K ? c + 1 : 0];  // rank c+1's first gradient
  const size_t chunk0 = (size_t)c * p.C;
  float* o32 = W32 ? p.out32[c] : nullptr;
  uint16_t* o16 = W16 ? p.out16[c] : nullptr;
  float* carry = MODE != kSettleWhole ? p.carry[c] : nullptr;
  const size_t T = (size_t)gridDim.x * kThreads;
  for (size_t u = (size_t)blockIdx.x * kThreads + threadIdx.x; u < p.units; u += T) {
    const size_t off = chunk0 + u * 8;
    uint4 rc[2];
    if constexpr (MODE == kSettleMiddle || MODE == kSettleLast)
      Vec8<float>::load_rw(carry + u * 8, rc);
    float total[8], acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) total[e] = acc[e] = 0.0f;
    for (int i0 = 0; i0 < n; i0 += B) {
      uint4 raw[B][L];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (i0 + b < n) {
          int idx = s0 + i0 + b;
          if (idx >= n) idx -= n;
          Vec8<Tg>::load(static_cast<const Tg*>(p.items[idx]) + off, raw[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (i0 + b < n) {
          int idx = s0 + i0 + b;
          if (idx >= n) idx -= n;
          if (p.first[idx]) {  // a new rank: its predecessor's accumulator joins the total
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              total[e] = __fadd_rn(total[e], acc[e]);
              acc[e] = 0.0f;
            }
          }
          float v[8];
          Vec8<Tg>::widen(raw[b], v);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], v[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) total[e] = __fadd_rn(total[e], acc[e]);  // the settled chunk
    if constexpr (MODE == kSettleFirst) {
#pragma unroll
      for (int e = 0; e < 8; ++e) total[e] = __fadd_rn(0.0f, total[e]);
      store8_f32(carry + u * 8, total);
    } else {
      if constexpr (MODE == kSettleMiddle || MODE == kSettleLast) {
        float cv[8];
        Vec8<float>::widen(rc, cv);
#pragma unroll
        for (int e = 0; e < 8; ++e) total[e] = __fadd_rn(cv[e], total[e]);
      }
      if constexpr (MODE == kSettleMiddle) {
        store8_f32(carry + u * 8, total);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) total[e] = __fmul_rn(total[e], p.scale);
        if (W32) store8_f32(o32 + u * 8, total);
        if (W16) store8_bf16(o16 + u * 8, total);
      }
    }
  }
}

template <typename Tg>
__global__ void __launch_bounds__(kThreads) odc_scalar_kernel(const __grid_constant__ OdcParams p) {
  const int c = blockIdx.y;
  const int K = p.K;
  const size_t chunk0 = (size_t)c * p.C;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < p.C;
       i += (size_t)gridDim.x * kThreads) {
    float total = 0.0f;
    for (int jr = 0; jr < K; ++jr) {
      const int q = ring_rank(c, jr, K);
      float acc = 0.0f;
      for (int j = 0; j < p.m[q]; ++j) {
        const Tg* gp = static_cast<const Tg*>(p.grads[q][j]);
        if (gp) acc = __fadd_rn(acc, widen_scalar(gp, chunk0 + i));
      }
      total = (jr == 0) ? acc : __fadd_rn(total, acc);
    }
    if (p.mode == kSettleFirst) {
      p.carry[c][i] = __fadd_rn(0.0f, total);
      continue;
    }
    if (p.mode == kSettleMiddle || p.mode == kSettleLast) {
      total = __fadd_rn(p.carry[c][i], total);
      if (p.mode == kSettleMiddle) {
        p.carry[c][i] = total;
        continue;
      }
    }
    total = __fmul_rn(total, p.scale);
    if (p.out32[c]) p.out32[c][i] = total;
    if (p.out16[c]) p.out16[c][i] = bf16_rn(total);
  }
}

template <typename Tg, bool FIRST, bool HAS_G>
cudaError_t acc_launch_k(const AccParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  const int occ = occupancy_blocks(acc_vec_kernel<Tg, FIRST, HAS_G>, dev.device);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x(dev.sm_count, occ, 1, p.units + 1, kThreads), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, acc_vec_kernel<Tg, FIRST, HAS_G>, p);
}

template <typename Tg>
cudaError_t acc_launch_t(const AccParams& p, bool first, bool vec, const dph::DeviceInfo& dev,
                         cudaStream_t s) {
  if (!vec) {
    const int occ = occupancy_blocks(acc_scalar_kernel<Tg>, dev.device);
    dim3 grid(grid_x(dev.sm_count, occ, 1, p.N, kThreads), 1);
    acc_scalar_kernel<Tg><<<grid, kThreads, 0, s>>>(p, first ? 1 : 0);
    return cudaGetLastError();
  }
  const bool has_g = p.grad != nullptr;
  if (first && has_g) return acc_launch_k<Tg, true, true>(p, dev, s);
  if (first) return acc_launch_k<Tg, true, false>(p, dev, s);
  if (has_g) return acc_launch_k<Tg, false, true>(p, dev, s);
  return acc_launch_k<Tg, false, false>(p, dev, s);
}

// CTAs per chunk for a settle launch: the shared sizing (which applies the
// process-wide limit), further capped by this launch's own limit if any.
inline unsigned odc_grid_x(int sm_count, int occ, int chunks, size_t work_items, int cta_limit) {
  unsigned gx = grid_x(sm_count, occ, chunks, work_items, kThreads);
  if (cta_limit > 0) {
    const unsigned cap = (unsigned)std::max(1, (cta_limit + chunks - 1) / chunks);
    gx = std::min(gx, cap);
  }
  return gx;
}

template <typename Tg, int MODE>
void (*odc_vec_pick(bool w32, bool w16))(OdcParams) {
  if (w32 && w16) return odc_vec_kernel<Tg, true, true, MODE>;
  if (w32) return odc_vec_kernel<Tg, true, false, MODE>;
  return odc_vec_kernel<Tg, false, true, MODE>;
}

template <typename Tg>
cudaError_t odc_launch_t(const OdcParams& p, bool w32, bool w16, bool vec, int cta_limit,
                         const dph::DeviceInfo& dev, cudaStream_t s) {
  if (!vec) {
    const int occ = occupancy_blocks(odc_scalar_kernel<Tg>, dev.device);
    dim3 grid(odc_grid_x(dev.sm_count, occ, p.K, p.C, cta_limit), p.K);
    odc_scalar_kernel<Tg><<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  void (*kern)(OdcParams);
  switch (p.mode) {
    case kSettleFirst: kern = odc_vec_kernel<Tg, false, false, kSettleFirst>; break;
    case kSettleMiddle: kern = odc_vec_kernel<Tg, false, false, kSettleMiddle>; break;
    case kSettleLast: kern = odc_vec_pick<Tg, kSettleLast>(w32, w16); break;
    default: kern = odc_vec_pick<Tg, kSettleWhole>(w32, w16); break;
  }
  const int occ = occupancy_blocks(kern, dev.device);
  dim3 grid(odc_grid_x(dev.sm_count, occ, p.K, p.units, cta_limit), p.K);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

namespace dpl {

cudaError_t launch_accumulate(const AccArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  AccParams p{};
  p.acc = a.acc;
  p.grad = a.grad;
  p.N = a.N;
  p.units = a.N / 8;
  if (a.grad_dtype == DP_FP32) return acc_launch_t<float>(p, a.first, a.vec_ok, dev, s);
  return acc_launch_t<uint16_t>(p, a.first, a.vec_ok, dev, s);
}

cudaError_t launch_odc_reduce_scatter(const OdcArgs& a, const dph::DeviceInfo& dev,
                                      cudaStream_t s) {
  OdcParams p{};
  int n = 0;
  for (int r = 0; r < a.K; ++r) {
    for (int j = 0; j < kMaxMb; ++j) p.grads[r][j] = a.grads[r][j];
    p.m[r] = a.m[r];
    p.out32[r] = a.out32[r];
    p.out16[r] = a.out16[r];
    p.pos[r] = n;
    bool first = true;
    for (int j = 0; j < a.m[r]; ++j) {
      if (!a.grads[r][j]) continue;  // a padding bucket adds +0
      p.items[n] = a.grads[r][j];
      p.first[n] = first ? 1 : 0;
      first = false;
      ++n;
    }
  }
  p.n_items = n;
  p.K = a.K;
  p.C = a.C;
  p.units = a.C / 8;
  p.scale = a.scale;
  // phase bits (first, last) -> what the launch does with the owners'
  // accumulators; first and last together is the whole minibatch at once
  const bool first = (a.phase & DP_SETTLE_FIRST) != 0, last = (a.phase & DP_SETTLE_LAST) != 0;
  p.mode = first && last ? kSettleWhole : first ? kSettleFirst : last ? kSettleLast
                                                                      : kSettleMiddle;
  for (int r = 0; r < a.K; ++r) p.carry[r] = p.mode == kSettleWhole ? nullptr : a.carry[r];
  const bool w32 = a.out32[0] != nullptr, w16 = a.out16[0] != nullptr;
  if (a.grad_dtype == DP_FP32)
    return odc_launch_t<float>(p, w32, w16, a.vec_ok, a.cta_limit, dev, s);
  return odc_launch_t<uint16_t>(p, w32, w16, a.vec_ok, a.cta_limit, dev, s);
}

}  // namespace dpl
