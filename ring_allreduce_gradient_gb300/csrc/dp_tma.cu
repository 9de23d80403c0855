// dp_tma.cu -- the all-reduce and all-gather streamed through shared memory
// with bulk asynchronous copies (cp.async.bulk, the 1-D form of TMA).
//
// The all-reduce of "CMU 11-868 L14-L15: Distributed Training and Data
// Parallelism, and Where Gradient Sync Costs Come From" (section "Ring
// AllReduce: ReduceScatter, then AllGather") touches every element of every
// rank twice: once to fold it into the chunk's ring-order sum, once to write
// the sum back.  Here each tile of a chunk is fetched from the K ranks by K
// bulk loads into shared memory, folded there by the CTA's threads (ring order
// x_{c+1} + ... + x_c in fp32, scale, cast) into an output tile, and written
// back to the K ranks by K bulk stores issued from one thread -- the data
// crosses shared memory once instead of passing through 16 store
// instructions per thread.  The all-gather is a copy pipeline without the
// fold: each CTA loads tiles of the gathered vector and stores them to one
// rank's buffer, the K ranks' CTAs reading each tile at the same time.
//
// Pipeline per CTA (one chunk, tiles strided over the CTAs of that chunk):
// loads run up to four tiles ahead in a ring of input tiles guarded by
// mbarriers (expect_tx); the output tile is double-buffered and released by
// cp.async.bulk.wait_group.read.  Every wait on an mbarrier is bounded; the
// threads of a CTA agree on an expiry with __syncthreads_or, so all of them
// leave the loop together, drain the copies in flight and return.

#include "dp_launch.h"

#include <algorithm>

namespace {

using namespace dpk;

constexpr uint64_t kTimeoutNs = 2000000000ull;

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__host__ __device__ __forceinline__ size_t min_sz(size_t a, size_t b) { return a < b ? a : b; }

__device__ __forceinline__ int ring_rank(int c, int j, int K) {
  int r = c + 1 + j;
  return r >= K ? r - K : r;
}

// ---------------------------------------------------------------------------
// All-reduce
// ---------------------------------------------------------------------------
constexpr int kArThreads = 256;
constexpr uint32_t kArTileBytes = 4096;  // per rank; 16 bytes per thread
// Input tile ring: 5 stages with 4 tiles in flight up to K=8 (measured on
// GB300: 3/2 gave 6.32, 4/3 6.73, 5/4 6.76, 6/5 6.76 TB/s at K=8 x 256 MiB);
// K=16 tiles are twice as large, so 3 stages with 2 in flight fit in 227 KB.
// Each rank's tile is 4 KiB x kVec (kVec 16-byte vectors per thread), so a
// stage always holds 32 KiB or more whatever K (K=2 and K=4 would otherwise
// pay a barrier per 8 or 16 KiB).
template <int KMAX>
struct ArDepth {
  static constexpr int kStages = KMAX <= 8 ? 5 : 3;
  static constexpr int kAhead = kStages - 1;
  static constexpr int kVec = KMAX >= 8 ? 1 : 8 / KMAX;
  static constexpr uint32_t kRankBytes = kArTileBytes * kVec;
};

struct ArTmaParams {
  void* bufs[kMaxK];
  int K;
  size_t N;
  size_t C;
  float scale;
  unsigned* err;
};

template <typename T>
struct Pack16;  // 16 bytes of T <-> fp32
template <>
struct Pack16<float> {
  static constexpr int E = 4;
  __device__ __forceinline__ static void widen(uint4 v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 narrow(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};
template <>
struct Pack16<uint16_t> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void widen(uint4 v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
  }
  __device__ __forceinline__ static uint4 narrow(const float (&f)[8]) {
    return make_uint4(pack_bf16x2_rn(f[0], f[1]), pack_bf16x2_rn(f[2], f[3]),
                      pack_bf16x2_rn(f[4], f[5]), pack_bf16x2_rn(f[6], f[7]));
  }
};

__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(uint16_t* p, float v) { *p = bf16_rn(v); }

template <typename T, int KMAX>
__global__ void __launch_bounds__(kArThreads) ar_tma_kernel(const __grid_constant__ ArTmaParams p) {
  constexpr int E = Pack16<T>::E;  // elements per 16 bytes
  constexpr int kArStages = ArDepth<KMAX>::kStages;
  constexpr int kArAhead = ArDepth<KMAX>::kAhead;
  constexpr int V = ArDepth<KMAX>::kVec;
  constexpr uint32_t RB = ArDepth<KMAX>::kRankBytes;  // bytes of one rank's tile
  constexpr uint32_t TILE = RB / sizeof(T);           // elements per rank tile
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* in_tiles = smem;                                   // [S][K][RB]
  unsigned char* out_tiles = smem + (size_t)kArStages * KMAX * RB;  // [2][RB]
  uint64_t* full = reinterpret_cast<uint64_t*>(out_tiles + 2 * RB);
  const int K = p.K;
  const int c = blockIdx.y;
  const size_t chunk0 = (size_t)c * p.C;
  if (chunk0 >= p.N) return;
  const size_t len = (p.N - chunk0) < p.C ? (p.N - chunk0) : p.C;
  const size_t vlen = len / 8 * 8;  // bulk-copied part; the rest is the scalar tail
  const size_t ntiles = (vlen + TILE - 1) / TILE;
  const size_t my_tiles =
      blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kArStages; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  auto tile_of = [&](size_t i) { return (size_t)blockIdx.x + i * gridDim.x; };
  auto issue_load = [&](size_t i) {  // thread 0
    const int s = (int)(i % kArStages);
    const size_t e0 = tile_of(i) * TILE;
    const uint32_t n = (uint32_t)min_sz(TILE, vlen - e0);
    mbar_arrive_expect_tx(&full[s], n * (uint32_t)sizeof(T) * (uint32_t)K);
    for (int j = 0; j < K; ++j)
      bulk_load(in_tiles + ((size_t)s * KMAX + j) * RB,
                static_cast<const T*>(p.bufs[ring_rank(c, j, K)]) + chunk0 + e0,
                n * (uint32_t)sizeof(T), &full[s]);
  };

  if (threadIdx.x == 0)
    for (size_t i = 0; i < (size_t)kArAhead && i < my_tiles; ++i) issue_load(i);

  size_t issued = min_sz(kArAhead, my_tiles);
  size_t i = 0;  // tiles consumed
  for (; i < my_tiles; ++i) {
    const int s = (int)(i % kArStages);
    const int ob = (int)(i & 1);
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((i / kArStages) & 1), p.err,
                                      kTimeoutNs);
    if (threadIdx.x == 0) bulk_wait_read<1>();  // output tile `ob` (two tiles ago) is free
    if (__syncthreads_or(!ok)) break;
    const size_t e0 = tile_of(i) * TILE;
    const uint32_t n = (uint32_t)min_sz(TILE, vlen - e0);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const uint32_t my = (threadIdx.x + v * kArThreads) * E;
      if (my < n) {
        float acc[E];
        Pack16<T>::widen(*reinterpret_cast<const uint4*>(in_tiles + (size_t)s * KMAX * RB +
                                                         my * sizeof(T)),
                         acc);
#pragma unroll
        for (int j = 1; j < KMAX; ++j) {
          if (j < K) {
            float x[E];
            Pack16<T>::widen(*reinterpret_cast<const uint4*>(
                                 in_tiles + ((size_t)s * KMAX + j) * RB + my * sizeof(T)),
                             x);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
          }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = __fmul_rn(acc[e], p.scale);
        *reinterpret_cast<uint4*>(out_tiles + (size_t)ob * RB + my * sizeof(T)) =
            Pack16<T>::narrow(acc);
      }
    }
    fence_proxy_async_smem();  // generic-proxy writes -> visible to the bulk stores
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int j = 0; j < K; ++j)
        bulk_store(static_cast<T*>(p.bufs[j]) + chunk0 + e0, out_tiles + (size_t)ob * RB,
                   n * (uint32_t)sizeof(T));
      bulk_commit();
      if (issued < my_tiles) {
        issue_load(issued);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) {
    bulk_wait_all();
    // Loads issued but never consumed (only after an expiry): at most
    // kArAhead of them, each the latest phase of a distinct stage, so a
    // parity wait on each is well defined.  Bounded.
    for (size_t t = i; t < issued; ++t)
      (void)mbar_wait_bounded(&full[t % kArStages], (uint32_t)((t / kArStages) & 1), p.err,
                              kTimeoutNs);
  }
  // ragged tail of the chunk (fewer than 8 elements), after the bulk part
  if (blockIdx.x == 0) {
    __syncthreads();
    for (size_t i = vlen + threadIdx.x; i < len; i += kArThreads) {
      float acc = widen_scalar(static_cast<const T*>(p.bufs[ring_rank(c, 0, K)]), chunk0 + i);
      for (int j = 1; j < K; ++j)
        acc = __fadd_rn(acc, widen_scalar(static_cast<const T*>(p.bufs[ring_rank(c, j, K)]),
                                          chunk0 + i));
      acc = __fmul_rn(acc, p.scale);
      for (int j = 0; j < K; ++j) store1(static_cast<T*>(p.bufs[j]) + chunk0 + i, acc);
    }
  }
}

template <int KMAX>
constexpr size_t ar_smem_bytes() {
  return (size_t)ArDepth<KMAX>::kStages * KMAX * ArDepth<KMAX>::kRankBytes +
         2 * ArDepth<KMAX>::kRankBytes + 64;
}

// ---------------------------------------------------------------------------
// Reduce-scatter: the same tile pipeline, the folded tile written once to the
// owner's shard (fp32 and/or bf16) by bulk stores.
// ---------------------------------------------------------------------------
constexpr int kRsThreads = 256;
// Input ring depth: 4 stages (3 tiles in flight) up to K=8; K=16 tiles are
// twice as large, so 2 stages keep the footprint under 227 KB.
template <int KMAX>
struct RsDepth {
  static constexpr int kStages = KMAX <= 8 ? 4 : 2;
  static constexpr int kAhead = kStages - 1;
};

struct RsTmaParams {
  const void* in[kMaxK];
  float* out32[kMaxK];
  uint16_t* out16[kMaxK];
  int K;
  size_t C;  // chunk length (N / K), a multiple of 8
  float scale;
  unsigned* err;
};

template <typename T, int KMAX, bool W32, bool W16>
__global__ void __launch_bounds__(kRsThreads) rs_tma_kernel(const __grid_constant__ RsTmaParams p) {
  constexpr int E = Pack16<T>::E;
  constexpr uint32_t TILE = kArTileBytes / sizeof(T);      // elements per rank tile
  constexpr uint32_t O32 = W32 ? TILE * 4 : 0;              // output tile bytes
  constexpr uint32_t O16 = W16 ? TILE * 2 : 0;
  constexpr int kRsStages = RsDepth<KMAX>::kStages;
  constexpr int kRsAhead = RsDepth<KMAX>::kAhead;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* in_tiles = smem;                                             // [S][K][4096]
  unsigned char* out_tiles = smem + (size_t)kRsStages * KMAX * kArTileBytes;  // [2][O32 + O16]
  uint64_t* full = reinterpret_cast<uint64_t*>(out_tiles + 2 * (O32 + O16));
  const int K = p.K;
  const int c = blockIdx.y;
  const size_t chunk0 = (size_t)c * p.C;
  const size_t ntiles = (p.C + TILE - 1) / TILE;
  const size_t my_tiles =
      blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRsStages; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  auto tile_of = [&](size_t i) { return (size_t)blockIdx.x + i * gridDim.x; };
  auto issue_load = [&](size_t i) {  // thread 0
    const int s = (int)(i % kRsStages);
    const size_t e0 = tile_of(i) * TILE;
    const uint32_t n = (uint32_t)min_sz(TILE, p.C - e0);
    mbar_arrive_expect_tx(&full[s], n * (uint32_t)sizeof(T) * (uint32_t)K);
    for (int j = 0; j < K; ++j)
      bulk_load(in_tiles + ((size_t)s * KMAX + j) * kArTileBytes,
                static_cast<const T*>(p.in[ring_rank(c, j, K)]) + chunk0 + e0,
                n * (uint32_t)sizeof(T), &full[s]);
  };

  size_t issued = min_sz(kRsAhead, my_tiles);
  if (threadIdx.x == 0)
    for (size_t i = 0; i < issued; ++i) issue_load(i);

  size_t i = 0;  // tiles consumed
  for (; i < my_tiles; ++i) {
    const int s = (int)(i % kRsStages);
    unsigned char* ob = out_tiles + (size_t)(i & 1) * (O32 + O16);
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((i / kRsStages) & 1), p.err,
                                      kTimeoutNs);
    if (threadIdx.x == 0) bulk_wait_read<1>();  // output tile of two tiles ago is free
    if (__syncthreads_or(!ok)) break;
    const size_t e0 = tile_of(i) * TILE;
    const uint32_t n = (uint32_t)min_sz(TILE, p.C - e0);
    const uint32_t my = threadIdx.x * E;
    if (my < n) {
      float acc[E];
      Pack16<T>::widen(*reinterpret_cast<const uint4*>(in_tiles + (size_t)s * KMAX * kArTileBytes +
                                                       my * sizeof(T)),
                       acc);
#pragma unroll
      for (int j = 1; j < KMAX; ++j) {
        if (j < K) {
          float v[E];
          Pack16<T>::widen(*reinterpret_cast<const uint4*>(
                               in_tiles + ((size_t)s * KMAX + j) * kArTileBytes + my * sizeof(T)),
                           v);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = __fadd_rn(acc[e], v[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = __fmul_rn(acc[e], p.scale);
      if (W32) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q)
          *reinterpret_cast<uint4*>(ob + (size_t)(my + 4 * q) * 4) =
              make_uint4(__float_as_uint(acc[4 * q]), __float_as_uint(acc[4 * q + 1]),
                         __float_as_uint(acc[4 * q + 2]), __float_as_uint(acc[4 * q + 3]));
      }
      if (W16) {
        unsigned char* o16 = ob + O32 + (size_t)my * 2;
        if (E == 8) {
          *reinterpret_cast<uint4*>(o16) =
              make_uint4(pack_bf16x2_rn(acc[0], acc[1]), pack_bf16x2_rn(acc[2], acc[3]),
                         pack_bf16x2_rn(acc[4 % E], acc[5 % E]),
                         pack_bf16x2_rn(acc[6 % E], acc[7 % E]));
        } else {
          *reinterpret_cast<uint2*>(o16) =
              make_uint2(pack_bf16x2_rn(acc[0], acc[1]), pack_bf16x2_rn(acc[2], acc[3]));
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      if (W32) bulk_store(p.out32[c] + e0, ob, n * 4u);
      if (W16) bulk_store(p.out16[c] + e0, ob + O32, n * 2u);
      bulk_commit();
      if (issued < my_tiles) {
        issue_load(issued);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) {
    bulk_wait_all();
    for (size_t t = i; t < issued; ++t)
      (void)mbar_wait_bounded(&full[t % kRsStages], (uint32_t)((t / kRsStages) & 1), p.err,
                              kTimeoutNs);
  }
}

template <typename T, int KMAX, bool W32, bool W16>
constexpr size_t rs_smem_bytes() {
  return (size_t)RsDepth<KMAX>::kStages * KMAX * kArTileBytes +
         2 * ((W32 ? (kArTileBytes / sizeof(T)) * 4 : 0) + (W16 ? (kArTileBytes / sizeof(T)) * 2 : 0)) +
         64;
}

// ---------------------------------------------------------------------------
// DDP bucket all-reduce through shared memory.  Tiles run over each tensor's
// 16-byte-aligned body (its first numel/8*8 elements); a tile's K rank copies
// land in rank-ordered slots, and each 16-byte vector is folded in the ring
// order of its chunk of the flattened bucket (chunk = bucket offset / C), or
// element by element where a chunk boundary splits the vector.  The <8
// trailing elements of each tensor are folded by block 0 at the end.
// ---------------------------------------------------------------------------
constexpr int kMtTmaMax = 96;  // tensors per launch (kernel parameter space)

struct MtTmaParams {
  void* ptr[kMtTmaMax][kMaxK];
  unsigned long long off[kMtTmaMax];    // bucket offset of the tensor's first element
  unsigned long long numel[kMtTmaMax];
  unsigned tstart[kMtTmaMax + 1];       // prefix sums of tiles per tensor
  int n, K;
  unsigned long long C;                 // chunk length of the whole bucket
  float scale;
  unsigned* err;
};

template <typename T, int KMAX>
__global__ void __launch_bounds__(kArThreads) mt_tma_kernel(const __grid_constant__ MtTmaParams p) {
  // Launched with programmatic stream serialization: this grid may be
  // scheduled while the previous kernel of the stream is still draining.
  // Let the next bucket's grid start scheduling onto SMs this one frees, set
  // up the barriers, then wait until the previous kernel has completed and
  // its writes are visible before touching global memory (a no-op after a
  // kernel that does not allow it).  Setting up first: 1 MiB buckets
  // 1.380 -> 1.368 ms per GPT-2-small iteration.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int E = Pack16<T>::E;
  constexpr int kStages = ArDepth<KMAX>::kStages;
  constexpr int kAhead = ArDepth<KMAX>::kAhead;
  constexpr int V = ArDepth<KMAX>::kVec;
  constexpr uint32_t RB = ArDepth<KMAX>::kRankBytes;
  constexpr uint32_t TILE = RB / sizeof(T);
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* in_tiles = smem;                                 // [S][K][RB], slot = rank
  unsigned char* out_tiles = smem + (size_t)kStages * KMAX * RB;  // [2][RB]
  uint64_t* full = reinterpret_cast<uint64_t*>(out_tiles + 2 * RB);
  const int K = p.K;
  const unsigned ntiles = p.tstart[p.n];
  const size_t my_tiles =
      blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // A CTA's tiles come in increasing order, so each side (the loads issued
  // ahead by thread 0, the tile being folded) keeps a tensor cursor that only
  // moves forward, and thread 0 keeps the current tensor's K pointers in
  // registers for each side -- the per-tensor tables in the kernel parameters
  // are read once per tensor, not once per tile.
  // A cursor also tracks the chunk of its tile's first element (ct) and the
  // next chunk boundary (nb); bucket offsets only grow, so both advance by
  // comparison, with one division on the first tile.
  struct Cursor {
    int t = 0;
    size_t e0 = 0;
    uint32_t n = 0;
    int ct = -1;
    unsigned long long nb = 0;
  };
  auto advance = [&](Cursor& cu, size_t i) {
    const unsigned g = (unsigned)((size_t)blockIdx.x + i * gridDim.x);
    while (cu.t + 1 < p.n && p.tstart[cu.t + 1] <= g) ++cu.t;
    cu.e0 = (size_t)(g - p.tstart[cu.t]) * TILE;
    const size_t body = p.numel[cu.t] / 8 * 8;
    cu.n = (uint32_t)min_sz(TILE, body - cu.e0);
    const unsigned long long tb = p.off[cu.t] + cu.e0;
    if (cu.ct < 0) {
      cu.ct = (int)(tb / p.C);
      cu.nb = (unsigned long long)(cu.ct + 1) * p.C;
    }
    while (tb >= cu.nb) {
      ++cu.ct;
      cu.nb += p.C;
    }
  };
  Cursor ld, cm;  // load side (thread 0), fold side (every thread)
  int ld_t = -1, ld_ct = -1, st_t = -1;
  const T* ld_rot[KMAX];  // rank pointers of the load-side tensor, in fold order of ld_ct
  T* st_ptr[KMAX];
  auto issue_load = [&](size_t i) {  // thread 0
    advance(ld, i);
    if (ld.t != ld_t || ld.ct != ld_ct) {
      ld_t = ld.t;
      ld_ct = ld.ct;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        ld_rot[j] = j < K ? static_cast<const T*>(p.ptr[ld_t][ring_rank(ld_ct, j, K)]) : nullptr;
    }
    const int s = (int)(i % kStages);
    // slot j holds rank ring_rank(ct, j): the fold order of the chunk of the
    // tile's first element (a vector of the next chunk shifts by one slot)
    mbar_arrive_expect_tx(&full[s], ld.n * (uint32_t)sizeof(T) * (uint32_t)K);
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K)
        bulk_load(in_tiles + ((size_t)s * KMAX + j) * RB, ld_rot[j] + ld.e0,
                  ld.n * (uint32_t)sizeof(T), &full[s]);
  };

  if (threadIdx.x == 0)
    for (size_t i = 0; i < (size_t)kAhead && i < my_tiles; ++i) issue_load(i);

  size_t issued = min_sz(kAhead, my_tiles);
  size_t i = 0;  // tiles consumed
  for (; i < my_tiles; ++i) {
    const int s = (int)(i % kStages);
    const int ob = (int)(i & 1);
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((i / kStages) & 1), p.err, kTimeoutNs);
    if (threadIdx.x == 0) bulk_wait_read<1>();
    if (__syncthreads_or(!ok)) break;
    advance(cm, i);
    const int t = cm.t;
    const size_t e0 = cm.e0;
    const uint32_t n = cm.n;
    const unsigned char* slots = in_tiles + (size_t)s * KMAX * RB;
    // Chunk of the tile's first element and the next chunk boundary: when a
    // chunk is at least a tile long a tile holds at most one boundary, so the
    // per-vector chunk is a comparison, not a 64-bit division.
    const unsigned long long tb = p.off[t] + e0;
    const bool one_boundary = p.C >= TILE;
    const int ct = cm.ct;  // the chunk the slots are rotated for
    const unsigned long long next_b = cm.nb;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const uint32_t my = (threadIdx.x + v * kArThreads) * E;
      if (my < n) {
        const unsigned long long b0 = tb + my;  // bucket offset of the vector
        const int c0 = one_boundary ? ct + (b0 >= next_b ? 1 : 0) : (int)(b0 / p.C);
        const int c1 = one_boundary ? ct + (b0 + E - 1 >= next_b ? 1 : 0)
                                    : (int)((b0 + E - 1) / p.C);
        // slot of fold position j for chunk c: (j + c - ct) mod K
        auto slot = [&](int j, int c) {
          int q = j + (c - ct) % K;
          return q >= K ? q - K : q;
        };
        float out[E];
        if (c0 == c1 && c0 == ct) {  // the common case: constant slot offsets
          Pack16<T>::widen(*reinterpret_cast<const uint4*>(slots + my * sizeof(T)), out);
#pragma unroll
          for (int j = 1; j < KMAX; ++j) {
            if (j < K) {
              float x[E];
              Pack16<T>::widen(
                  *reinterpret_cast<const uint4*>(slots + (size_t)j * RB + my * sizeof(T)), x);
#pragma unroll
              for (int e = 0; e < E; ++e) out[e] = __fadd_rn(out[e], x[e]);
            }
          }
        } else if (c0 == c1) {
          Pack16<T>::widen(*reinterpret_cast<const uint4*>(
                               slots + (size_t)slot(0, c0) * RB + my * sizeof(T)),
                           out);
          for (int j = 1; j < K; ++j) {
            float x[E];
            Pack16<T>::widen(*reinterpret_cast<const uint4*>(
                                 slots + (size_t)slot(j, c0) * RB + my * sizeof(T)),
                             x);
#pragma unroll
            for (int e = 0; e < E; ++e) out[e] = __fadd_rn(out[e], x[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int ce = (int)((b0 + e) / p.C);
            float acc = 0.0f;
            for (int j = 0; j < K; ++j) {
              float x[E];
              Pack16<T>::widen(*reinterpret_cast<const uint4*>(
                                   slots + (size_t)slot(j, ce) * RB + my * sizeof(T)),
                               x);
              acc = j == 0 ? x[e] : __fadd_rn(acc, x[e]);
            }
            out[e] = acc;
          }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = __fmul_rn(out[e], p.scale);
        *reinterpret_cast<uint4*>(out_tiles + (size_t)ob * RB + my * sizeof(T)) =
            Pack16<T>::narrow(out);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      if (t != st_t) {
        st_t = t;
#pragma unroll
        for (int r = 0; r < KMAX; ++r) st_ptr[r] = r < K ? static_cast<T*>(p.ptr[st_t][r]) : nullptr;
      }
#pragma unroll
      for (int r = 0; r < KMAX; ++r)
        if (r < K)
          bulk_store(st_ptr[r] + e0, out_tiles + (size_t)ob * RB, n * (uint32_t)sizeof(T));
      bulk_commit();
      if (issued < my_tiles) {
        issue_load(issued);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) {
    bulk_wait_all();
    for (size_t u = i; u < issued; ++u)
      (void)mbar_wait_bounded(&full[u % kStages], (uint32_t)((u / kStages) & 1), p.err,
                              kTimeoutNs);
  }
  // the <8 trailing elements of every tensor of this launch
  if (blockIdx.x == 0) {
    __syncthreads();
    for (int t = 0; t < p.n; ++t) {
      const size_t body = p.numel[t] / 8 * 8;
      for (size_t e = body + threadIdx.x; e < p.numel[t]; e += kArThreads) {
        const int c = (int)((p.off[t] + e) / p.C);
        float acc = widen_scalar(static_cast<const T*>(p.ptr[t][ring_rank(c, 0, K)]), e);
        for (int j = 1; j < K; ++j)
          acc = __fadd_rn(acc, widen_scalar(static_cast<const T*>(p.ptr[t][ring_rank(c, j, K)]), e));
        acc = __fmul_rn(acc, p.scale);
        for (int j = 0; j < K; ++j) store1(static_cast<T*>(p.ptr[t][j]) + e, acc);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// All-gather
// ---------------------------------------------------------------------------
// Two schedules, both 64 KiB tiles in a 3-stage ring driven by one thread.
//
// One destination per CTA (the whole GPU): CTA (x, j) walks tiles x, x + G,
// ... of the gathered vector (shard 0's tiles, then shard 1's, ...), loads
// each from its shard and stores it to rank j's buffer, two loads ahead.  The
// K CTAs that share an x walk the same tiles at the same time, so a tile
// comes from DRAM once and from L2 for the other K - 1 ranks, and every CTA
// runs the plain copy pattern of one load and one store per tile.
//
// One source shard per CTA (a launch capped to part of the GPU): CTA (x, c)
// walks shard c's tiles and stores each to all K ranks, one load ahead.  On
// few SMs the per-CTA issue rate sets the pace, and K stores per load move
// more bytes per issued copy.
//
// Measured on GB300, 8 x 32 MiB -> 8 x 256 MiB on all SMs: one source shard
// per CTA 6.11-6.16 TB/s; one destination, one / two loads ahead 4.68 /
// 6.59-6.63; 2 / 4 / 8 destinations per CTA 5.35 / 5.89 / 6.11; 32 KiB and
// 16 KiB tiles 5.33-5.44.  8 x 16 MiB on 16 / 38 / 76 SMs: one source shard
// per CTA 1.151 / 0.483 / 0.259 ms, one destination 1.279 / 0.643 / 0.319 ms.
constexpr int kAgStages = 3;
constexpr uint32_t kAgTileBytes = 65536;
constexpr size_t kAgSmem = (size_t)kAgStages * kAgTileBytes + 64;

struct AgTmaParams {
  const unsigned char* shards[kMaxK];
  unsigned char* out[kMaxK];
  int K;
  size_t bytes;  // per shard, a multiple of 16
  size_t tps;    // tiles per shard (the last one may be short)
  unsigned* err;
};

template <bool kOneDest>
__global__ void __launch_bounds__(32) ag_tma_kernel(const __grid_constant__ AgTmaParams p) {
  constexpr int kAhead = kOneDest ? 2 : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kAgStages * kAgTileBytes);
  if (threadIdx.x != 0) return;  // one thread drives the copies of this CTA
  const int y = blockIdx.y;      // destination rank (kOneDest) or source shard
  const size_t ntiles = kOneDest ? p.tps * (size_t)p.K : p.tps;
  const size_t my_tiles =
      blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  for (int s = 0; s < kAgStages; ++s) mbar_init(&full[s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // tile i of this CTA: source shard and byte offset within it
  auto tile_of = [&](size_t i) { return (size_t)blockIdx.x + i * gridDim.x; };
  auto shard_of = [&](size_t i) { return kOneDest ? tile_of(i) / p.tps : (size_t)y; };
  auto off_of = [&](size_t i) {
    const size_t t = tile_of(i);
    return (kOneDest ? t - (t / p.tps) * p.tps : t) * kAgTileBytes;
  };
  auto size_of = [&](size_t i) { return (uint32_t)min_sz(kAgTileBytes, p.bytes - off_of(i)); };
  auto issue_load = [&](size_t i) {
    const int s = (int)(i % kAgStages);
    mbar_arrive_expect_tx(&full[s], size_of(i));
    bulk_load(smem + (size_t)s * kAgTileBytes, p.shards[shard_of(i)] + off_of(i), size_of(i),
              &full[s]);
  };
  size_t issued = 0;
  for (; issued < (size_t)kAhead && issued < my_tiles; ++issued) issue_load(issued);
  size_t i = 0;  // tiles consumed
  for (; i < my_tiles; ++i) {
    const int s = (int)(i % kAgStages);
    if (!mbar_wait_bounded(&full[s], (uint32_t)((i / kAgStages) & 1), p.err, kTimeoutNs)) break;
    const size_t dst = shard_of(i) * p.bytes + off_of(i);
    const unsigned char* src = smem + (size_t)s * kAgTileBytes;
    if (kOneDest) {
      bulk_store(p.out[y] + dst, src, size_of(i));
    } else {
      for (int j = 0; j < p.K; ++j) bulk_store(p.out[j] + dst, src, size_of(i));
    }
    bulk_commit();
    if (issued < my_tiles) {
      // the stage of tile `issued` last held tile issued-kAgStages = i+kAhead-kAgStages,
      // whose store group must be done reading it; the kAgStages-kAhead newer
      // groups may still be pending
      bulk_wait_read<kAgStages - kAhead>();
      issue_load(issued);
      ++issued;
    }
  }
  bulk_wait_all();
  // loads issued but never consumed (only after an expiry), bounded
  for (size_t t = i; t < issued; ++t)
    (void)mbar_wait_bounded(&full[t % kAgStages], (uint32_t)((t / kAgStages) & 1), p.err,
                            kTimeoutNs);
}

template <typename T, int KMAX>
cudaError_t ar_tma_launch_k(const ArTmaParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  constexpr size_t smem = ar_smem_bytes<KMAX>();
  const int occ = dph::prepare_kernel(reinterpret_cast<const void*>(ar_tma_kernel<T, KMAX>),
                                      kArThreads, smem, dev.device);
  if (occ < 1) return cudaErrorInvalidConfiguration;
  long long resident = (long long)dev.sm_count * occ;
  const int limit = dph::stream_cta_limit();
  if (limit > 0 && resident > limit) resident = limit;
  const size_t tile = ArDepth<KMAX>::kRankBytes / sizeof(T);
  long long per_chunk = (resident + p.K - 1) / p.K;
  long long need = (long long)((p.C + tile - 1) / tile);
  long long gx = std::max(1LL, std::min(per_chunk, need));
  ar_tma_kernel<T, KMAX><<<dim3((unsigned)gx, p.K), kArThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int KMAX>
cudaError_t mt_tma_launch_k(const MtTmaParams& p, unsigned tiles, const dph::DeviceInfo& dev,
                            cudaStream_t s) {
  constexpr size_t smem = ar_smem_bytes<KMAX>();
  const int occ = dph::prepare_kernel(reinterpret_cast<const void*>(mt_tma_kernel<T, KMAX>),
                                      kArThreads, smem, dev.device);
  if (occ < 1) return cudaErrorInvalidConfiguration;
  long long resident = (long long)dev.sm_count * occ;
  const int limit = dph::stream_cta_limit();
  if (limit > 0 && resident > limit) resident = limit;
  // at least one CTA, so block 0 folds the tensors' short tails
  long long gx = std::max(1LL, std::min<long long>(resident, (long long)tiles));
  // Back-to-back bucket launches overlap one grid's drain with the next one's
  // start-up (the kernel waits for its predecessor before any memory access).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gx, 1, 1);
  cfg.blockDim = dim3(kArThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mt_tma_kernel<T, KMAX>, p);
}

template <typename T, int KMAX, bool W32, bool W16>
cudaError_t rs_tma_launch_k(const RsTmaParams& p, const dph::DeviceInfo& dev, cudaStream_t s) {
  constexpr size_t smem = rs_smem_bytes<T, KMAX, W32, W16>();
  const int occ = dph::prepare_kernel(
      reinterpret_cast<const void*>(rs_tma_kernel<T, KMAX, W32, W16>), kRsThreads, smem,
      dev.device);
  if (occ < 1) return cudaErrorInvalidConfiguration;
  long long resident = (long long)dev.sm_count * occ;
  const int limit = dph::stream_cta_limit();
  if (limit > 0 && resident > limit) resident = limit;
  const size_t tile = kArTileBytes / sizeof(T);
  long long per_chunk = (resident + p.K - 1) / p.K;
  long long need = (long long)((p.C + tile - 1) / tile);
  long long gx = std::max(1LL, std::min(per_chunk, need));
  rs_tma_kernel<T, KMAX, W32, W16><<<dim3((unsigned)gx, p.K), kRsThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int KMAX>
cudaError_t rs_tma_launch_w(const RsTmaParams& p, bool w32, bool w16, const dph::DeviceInfo& dev,
                            cudaStream_t s) {
  if (w32 && w16) return rs_tma_launch_k<T, KMAX, true, true>(p, dev, s);
  if (w32) return rs_tma_launch_k<T, KMAX, true, false>(p, dev, s);
  return rs_tma_launch_k<T, KMAX, false, true>(p, dev, s);
}

template <typename T>
cudaError_t rs_tma_launch_t(const RsTmaParams& p, bool w32, bool w16, const dph::DeviceInfo& dev,
                            cudaStream_t s) {
  if (p.K <= 2) return rs_tma_launch_w<T, 2>(p, w32, w16, dev, s);
  if (p.K <= 4) return rs_tma_launch_w<T, 4>(p, w32, w16, dev, s);
  if (p.K <= 8) return rs_tma_launch_w<T, 8>(p, w32, w16, dev, s);
  return rs_tma_launch_w<T, 16>(p, w32, w16, dev, s);
}

}  // namespace

namespace dpl {

cudaError_t launch_reduce_scatter_tma(const RsArgs& a, const dph::DeviceInfo& dev,
                                      cudaStream_t s) {
  RsTmaParams p{};
  for (int r = 0; r < a.K; ++r) {
    p.in[r] = a.in[r];
    p.out32[r] = a.out32[r];
    p.out16[r] = a.out16[r];
  }
  p.K = a.K;
  p.C = a.C;
  p.scale = a.scale;
  p.err = dev.err_word;
  const bool w32 = a.out32[0] != nullptr, w16 = a.out16[0] != nullptr;
  if (a.in_dtype == DP_FP32) return rs_tma_launch_t<float>(p, w32, w16, dev, s);
  return rs_tma_launch_t<uint16_t>(p, w32, w16, dev, s);
}


cudaError_t launch_all_reduce_tma(const ArArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  ArTmaParams p{};
  for (int r = 0; r < a.K; ++r) p.bufs[r] = a.bufs[r];
  p.K = a.K;
  p.N = a.N;
  p.C = a.C;
  p.scale = a.scale;
  p.err = dev.err_word;
  const bool f32 = a.dtype == DP_FP32;
  if (a.K <= 2) return f32 ? ar_tma_launch_k<float, 2>(p, dev, s) : ar_tma_launch_k<uint16_t, 2>(p, dev, s);
  if (a.K <= 4) return f32 ? ar_tma_launch_k<float, 4>(p, dev, s) : ar_tma_launch_k<uint16_t, 4>(p, dev, s);
  if (a.K <= 8) return f32 ? ar_tma_launch_k<float, 8>(p, dev, s) : ar_tma_launch_k<uint16_t, 8>(p, dev, s);
  return f32 ? ar_tma_launch_k<float, 16>(p, dev, s) : ar_tma_launch_k<uint16_t, 16>(p, dev, s);
}

cudaError_t launch_bucket_allreduce_tma(const BucketArgs& a, const dph::DeviceInfo& dev,
                                        cudaStream_t s) {
  unsigned long long total = 0;
  for (int t = 0; t < a.n; ++t) total += a.numels[t];
  if (total == 0) return cudaSuccess;
  const unsigned long long C = (total + (unsigned long long)a.K - 1) / (unsigned long long)a.K;
  unsigned long long off = 0;
  int t = 0;
  while (t < a.n) {
    MtTmaParams p;
    memset(&p, 0, sizeof p);
    p.K = a.K;
    p.C = C;
    p.scale = a.scale;
    p.err = dev.err_word;
    const uint32_t RB = a.K <= 2 ? ArDepth<2>::kRankBytes
                        : a.K <= 4 ? ArDepth<4>::kRankBytes
                        : a.K <= 8 ? ArDepth<8>::kRankBytes
                                   : ArDepth<16>::kRankBytes;
    const unsigned long long tile = RB / (a.dtype == DP_FP32 ? 4u : 2u);
    int n = 0;
    unsigned tiles = 0;
    while (t < a.n && n < kMtTmaMax) {
      const unsigned long long ne = a.numels[t];
      const unsigned long long tt = (ne / 8 * 8 + tile - 1) / tile;
      if (n > 0 && (unsigned long long)tiles + tt > 0x7fffffffull) break;
      for (int r = 0; r < a.K; ++r) p.ptr[n][r] = a.ptrs[(size_t)t * a.K + r];
      p.off[n] = off;
      p.numel[n] = ne;
      p.tstart[n] = tiles;
      tiles += (unsigned)tt;
      off += ne;
      ++n;
      ++t;
    }
    p.n = n;
    p.tstart[n] = tiles;
    const bool f32 = a.dtype == DP_FP32;
    cudaError_t e;
    if (a.K <= 2) e = f32 ? mt_tma_launch_k<float, 2>(p, tiles, dev, s) : mt_tma_launch_k<uint16_t, 2>(p, tiles, dev, s);
    else if (a.K <= 4) e = f32 ? mt_tma_launch_k<float, 4>(p, tiles, dev, s) : mt_tma_launch_k<uint16_t, 4>(p, tiles, dev, s);
    else if (a.K <= 8) e = f32 ? mt_tma_launch_k<float, 8>(p, tiles, dev, s) : mt_tma_launch_k<uint16_t, 8>(p, tiles, dev, s);
    else e = f32 ? mt_tma_launch_k<float, 16>(p, tiles, dev, s) : mt_tma_launch_k<uint16_t, 16>(p, tiles, dev, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_all_gather_tma(const AgArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  AgTmaParams p{};
  for (int r = 0; r < a.K; ++r) {
    p.shards[r] = static_cast<const unsigned char*>(a.shards[r]);
    p.out[r] = static_cast<unsigned char*>(a.out[r]);
  }
  p.K = a.K;
  p.bytes = a.C * a.esz;
  p.tps = (p.bytes + kAgTileBytes - 1) / kAgTileBytes;
  p.err = dev.err_word;
  // both forms have the same shared memory and block size, so one occupancy
  const int occ = dph::prepare_kernel(reinterpret_cast<const void*>(ag_tma_kernel<true>), 32,
                                      kAgSmem, dev.device);
  if (occ < 1 || dph::prepare_kernel(reinterpret_cast<const void*>(ag_tma_kernel<false>), 32,
                                     kAgSmem, dev.device) < 1)
    return cudaErrorInvalidConfiguration;
  long long resident = (long long)dev.sm_count * occ;
  const int limit = dph::stream_cta_limit();
  const bool capped = limit > 0 && resident > limit;
  if (capped) resident = limit;
  if (!capped) {
    // K destinations x gx CTAs, all resident at once (rounding down, so that
    // no CTA waits for a second wave)
    long long gx = std::max(1LL, std::min(resident / a.K, (long long)(p.tps * (size_t)a.K)));
    ag_tma_kernel<true><<<dim3((unsigned)gx, a.K), 32, kAgSmem, s>>>(p);
  } else {
    long long gx = std::max(1LL, std::min((resident + a.K - 1) / a.K, (long long)p.tps));
    ag_tma_kernel<false><<<dim3((unsigned)gx, a.K), 32, kAgSmem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace dpl
