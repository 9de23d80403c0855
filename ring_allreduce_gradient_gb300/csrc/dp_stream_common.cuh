// dp_stream_common.cuh -- the pieces the HBM-streaming kernel files share:
// block size, the ring's rotated rank order, and grid sizing (a persistent
// grid of SMs x occupancy CTAs split over the chunks).
#pragma once

#include "dp_launch.h"

#include <algorithm>

namespace {

using namespace dpk;

constexpr int kThreads = 256;

// Rotated rank for position j of chunk c's fold: (c + 1 + j) mod K.
__device__ __forceinline__ int ring_rank(int c, int j, int K) {
  int r = c + 1 + j;
  return r >= K ? r - K : r;
}

// ---------------------------------------------------------------------------
// Grid sizing
// ---------------------------------------------------------------------------
template <typename KernelT>
int occupancy_blocks(KernelT kernel, int device) {
  const int b = dph::prepare_kernel(reinterpret_cast<const void*>(kernel), kThreads, 0, device);
  return b < 1 ? 1 : b;
}

// CTAs per chunk: the resident grid (SMs x occupancy) split over the chunks,
// never more than the chunk's work needs, at least one.
inline unsigned grid_x(int sm_count, int occ, int chunks, size_t work_items, int items_per_cta) {
  long long resident = (long long)sm_count * occ;
  const int limit = dph::stream_cta_limit();
  if (limit > 0 && resident > limit) resident = limit;
  long long per_chunk = (resident + chunks - 1) / chunks;
  long long need = (long long)((work_items + items_per_cta - 1) / items_per_cta);
  long long gx = std::min(per_chunk, need);
  if (gx < 1) gx = 1;
  if (gx > 65535LL * 1024) gx = 65535LL * 1024;
  return (unsigned)gx;
}

inline int kmax_for(int K) { return K <= 2 ? 2 : K <= 4 ? 4 : K <= 8 ? 8 : 16; }

}  // namespace
