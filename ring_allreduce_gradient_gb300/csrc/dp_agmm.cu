// dp_agmm.cu -- FSDP forward: the parameter all-gather fused into the local
// matmul, on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// "Sharding and Parallelism" (How to Scale Your Model on AMD, ch. 5), section
// "Real HLO before and after partitioning": each rank holds x[128,512] and a
// row shard w_k[64,512]; the partitioned program all-gathers w to w[512,512]
// and runs the local dot.  Section "FSDP and ZeRO": the forward pass gathers
// W before the dot.  Here the gathered weight is never materialised: each
// B tile of y = x . w^T is loaded by TMA straight from the shard(s) that hold
// its rows, through one tensor map per shard.
//
// Kernel structure (one persistent CTA per SM, 256 threads):
//   warps 0, 2  TMA producers, each filling alternate stages: A tile [128 x 64]
//               of x and B tile [BN x 64] of w per k-block into a 4-stage
//               shared-memory ring (128-byte swizzle), completion counted on
//               `full` mbarriers.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (kind::f16, bf16 x
//               bf16 -> fp32, M=128, N=BN, K=16) into one of two TMEM
//               accumulators; tcgen05.commit frees smem stages (`empty`) and
//               hands finished accumulators to the epilogue (`tmem_full`).
//   warp 2      also allocates / frees the 512 TMEM columns.
//   warps 4-7   epilogue: tcgen05.ld of 32 lanes x 16 columns at a time per
//               warp, scale, convert, store y (TMA stores from a swizzled
//               staging tile, or plain stores); then release the accumulator
//               (`tmem_empty`).
// Two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// An all-reduce-form problem with fewer tiles than half the CTAs gives each
// tile to 2, 4 or 8 CTAs ("copy groups"), each recomputing it and storing its
// share of the K output copies.
//
// Chained split of the last round (optional, with a caller's workspace):
// when the tiles fill the CTAs q times with R < CTAs/2 left over, the k-blocks
// of each of those R tiles are cut into s segments run by s different CTAs,
// each of which also runs q whole tiles.  A segment hands its fp32
// accumulator to the next one through the workspace (a release flag per
// hand-off); the next segment loads it back into TMEM and continues the same
// accumulation chain, so every output element sees exactly the MMAs it would
// see in one CTA and the result is bitwise the same with or without the
// split.  Segment j runs in slot q-s+1+j of its CTA's list (whole tiles
// before it: q-s+1+j), so it starts a whole tile after segment j-1 did, when
// that one has finished, and the CTAs stay in step until the last rounds.
//
// Every mbarrier wait is bounded (global timer); on expiry the waiting role
// flags the device error word, marks the CTA aborted and unwinds; the CTA
// drains what it issued (bounded) and frees TMEM before returning.

#include "dp_launch.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cstring>
#include <mutex>
#include <unordered_map>

namespace {

using namespace dpk;

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 elements in one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kMaxBN = 256;
constexpr int kAccCols = 256;   // TMEM columns per accumulator
constexpr int kTmemCols = 512;  // two accumulators
constexpr uint32_t kStageA = BM * BK * 2;      // 16 KiB
constexpr uint32_t kStageB = kMaxBN * BK * 2;  // 32 KiB
constexpr uint32_t kStageY = 16384;  // epilogue staging tile: 128 rows x 128 bytes
constexpr size_t kBarBytes = 256;
// One staging tile, not two: a second one measured no faster on GB300 (4(b)
// 168.0 against 168.7 us, TP all-reduce 238.4 against 238.3 us, weight
// gradient 180.3 both), and the 16 KiB it frees lets two 256-thread
// streaming CTAs (a settle running on another stream) share each SM with the
// GEMM's CTA: the settle pipeline of 32 layers went from 16.1 to 15.4 ms.
constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * (kStageA + kStageB) + (size_t)kStageY + kBarBytes;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s
constexpr int kMaxSplit = 4;     // segments per split tile
constexpr int kMinSegKb = 8;     // k-blocks per segment, at least
// TMA loads are issued by two warps, one for the even and one for the odd
// ring stages (kStages is even, so a stage's parity is its k-block's).
// Measured on GB300, one issuing warp completes about one box per ~770 SM
// clocks whatever its size up to 32 KiB, and more issuing warps add up
// (16 KiB boxes from an L2-resident tensor: 19 / 38 / 75 bytes per clock with
// 1 / 2 / 4 warps); one warp loading A and B for every 575-clock k-block
// would pace the MMAs.
constexpr int kProducerWarps = 2;
static_assert(kStages % kProducerWarps == 0, "stage parity must select the producer");
// Warps 0, 2 and 3 are free for producing (1 issues the MMAs, 4-7 drain
// TMEM); a fourth producer would be warp 8.
constexpr int kThreadsG = kProducerWarps > 3 ? 288 : 256;
__device__ __forceinline__ int producer_index(int warp) {
  const int i = warp == 0 ? 0 : (warp == 2 || warp == 3) ? warp - 1 : warp == 8 ? 3 : -1;
  return i < kProducerWarps ? i : -1;
}

// Operand sources.
//   kGatherB: A = x [M, D]; B row block f of the gathered w comes from shard
//             f / F_shard (the FSDP parameter all-gather).
//   kShardK:  rank r holds x_r [M, D_shard] and w_r [F, D_shard]; the k-blocks
//             of all ranks are chained into one accumulator, so the tensor
//             parallel psum of the partial products happens in TMEM.
//   kShardT:  the weight gradient.  Rank r holds dY_r [T, F] and X_r [T, D]
//             (tokens x features, row-major); the product is dW [F, D] =
//             sum_r dY_r^T X_r, so the contraction runs over tokens, which
//             are the rows of both operands: A = dY_r^T and B = X_r^T are read
//             MN-major, and the token blocks of all ranks chain into one
//             accumulator (the data-parallel psum of the per-rank dW_r).
//   kShardKxw: kShardK with each rank's weight in the x . w orientation,
//             w_r [D_shard, F] row-major (sharded along the contracted
//             rows): A = x_r K-major as in kShardK, B = w_r read MN-major as
//             in kShardT (a 3-D box of 64-column slabs of 64 rows of k).
enum { kGatherB = 0, kShardK = 1, kShardT = 2, kShardKxw = 3 };
// Output placement.
//   kOutOne:       y[0] [M, F]
//   kOutReplicate: the same [M, F] result into y[0..K-1] (all-reduce)
//   kOutRowShard:  rows [c*M/K, (c+1)*M/K) into y[c] (reduce-scatter of the
//                  flattened row-major result: chunk c of M*F elements)
enum { kOutOne = 0, kOutReplicate = 1, kOutRowShard = 2 };

struct AgmmParams {
  CUtensorMap tmA[kMaxK];
  CUtensorMap tmB[kMaxK];
  void* y[kMaxK];
  unsigned* err;
  int M, F, D;
  int F_shard;
  int BN;        // tile width along F (multiple of 16, <= 256)
  int box_rows;  // rows per B TMA box
  int boxes;     // BN / box_rows
  int tiles_m, tiles_n, num_kb;
  int y_f32;
  int mode;            // kGatherB / kShardK / kShardT / kShardKxw
  int kb_per_rank;     // kShardK(xw) / kShardT: k-blocks of one rank's D_shard / T
  int out_mode;        // kOutOne / kOutReplicate / kOutRowShard
  int K;               // ranks (outputs for kOutReplicate / kOutRowShard)
  int rows_per_shard;  // kOutRowShard: M / K
  float scale;         // applied to the fp32 accumulator before the cast
  int tma_epi;         // 1: stage output blocks in smem and store them with TMA
  int ec;              // epilogue column block (128 bytes of output per row)
  int out_evict_first; // TMA stores mark their L2 lines evict-first
  int dup;             // kOutReplicate: CTAs per output tile, each storing K / dup copies
  // chained split of the last round (split_s == 1: none)
  int split_s;         // segments per tail tile
  int split_q;         // whole tiles per CTA
  int split_R;         // tail tiles: the last R tile indices
  float* ws_part;      // partial accumulators, (s-1)*R blocks of [BN/16][128][16] fp32
  unsigned long long* ws_flag;  // one per partial block; == nonce once it is written
  unsigned long long nonce;     // this launch's flag value (never 0)
  CUtensorMap tmY[kMaxK];
};

// One CTA's work: tile `tile`, k-blocks [kb0, kb1); `load` / `store` name the
// partial block the accumulator starts from / is handed on through (-1: none).
struct Item {
  int tile, kb0, kb1, load, store;
  int grp;  // the tile's copy group (kOutReplicate with dup > 1), else 0
};

__device__ __forceinline__ int cta_items(const AgmmParams& p, int num_tiles) {
  const int b = blockIdx.x;
  if (p.split_s > 1) return p.split_q + (b < p.split_R * p.split_s ? 1 : 0);
  return b < num_tiles ? (num_tiles - 1 - b) / (int)gridDim.x + 1 : 0;
}

// Item w of this CTA.  Without a split: tiles b, b+G, b+2G, ...  With one:
// CTA b < R*s runs segment j = b / R of tail tile q*G + b % R at position
// q-s+1+j of its list and its q whole tiles b, b+G, ... around it.
__device__ __forceinline__ Item cta_item(const AgmmParams& p, int w) {
  const int b = blockIdx.x, G = gridDim.x;
  Item it{b + w * G, 0, p.num_kb, -1, -1, 0};
  if (p.dup > 1) {  // virtual tile v: tile v / dup, copy group v % dup (never split)
    it.grp = it.tile % p.dup;
    it.tile /= p.dup;
    return it;
  }
  if (p.split_s > 1 && b < p.split_R * p.split_s) {
    const int j = b / p.split_R, i = b - j * p.split_R;
    const int pos = p.split_q - (p.split_s - 1) + j;
    if (w == pos) {
      it.tile = p.split_q * G + i;
      it.kb0 = j * p.num_kb / p.split_s;
      it.kb1 = (j + 1) * p.num_kb / p.split_s;
      if (j > 0) it.load = (j - 1) * p.split_R + i;
      if (j + 1 < p.split_s) it.store = j * p.split_R + i;
    } else if (w > pos) {
      it.tile = b + (w - 1) * G;
    }
  }
  return it;
}

// ---- PTX wrappers ---------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// A 3-D box: (64 elements, rows, blocks of 64) -- the MN-major operand tiles
// of kShardT, viewed as (64 features, T tokens, features / 64).
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x,
                                             int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y)
      : "memory");
}

// The same store with an L2 policy: lines written under an evict-first policy
// are the first to leave L2, so a large output stream does not push out the
// operand tiles that other CTAs are still reading.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, const void* src, int x,
                                                  int y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Barrier 1 among the 128 epilogue threads; the reduction form makes every
// one of them take the same branch.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand laid out
// by TMA with the 128-byte swizzle; 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // bits 0-13: start address >> 4
  d |= (uint64_t)1u << 16;                   // bits 16-29: leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;         // bits 32-45: stride byte offset >> 4
  d |= (uint64_t)1u << 46;                   // bits 46-48: fixed 0b001
  d |= (uint64_t)2u << 61;                   // bits 61-63: 128-byte swizzle
  return d;
}

// The same for an MN-major operand (kShardT): TMA writes each 64-wide block
// of the M (or N) dimension as rows of 128 bytes, one row per k, 128-byte
// swizzled, the blocks 8 KiB apart (64 rows of k per stage).  Fields: the
// offset between those 64-wide blocks (bits 16-29) and between 8-row groups
// of k (bits 32-45).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // bits 0-13: start address >> 4
  d |= (uint64_t)(8192u >> 4) << 16;         // bits 16-29: next 64-wide M/N block
  d |= (uint64_t)(1024u >> 4) << 32;         // bits 32-45: next 8 rows of k
  d |= (uint64_t)1u << 46;                   // bits 46-48: fixed 0b001
  d |= (uint64_t)2u << 61;                   // bits 61-63: 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4)                        // D format: f32
         | (1u << 7)                      // A format: bf16
         | (1u << 10)                     // B format: bf16
         | ((uint32_t)(n >> 3) << 17)     // N >> 3
         | ((uint32_t)(m >> 4) << 24);    // M >> 4
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

#define DP_TMEM_LD_X16(taddr, r)                                                              \
  asm volatile(                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15}, [%16];"                                                                      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])                                                 \
      : "r"(taddr))

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

#define DP_TMEM_ST_X16(taddr, r)                                                              \
  asm volatile(                                                                               \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"  \
      "%13,%14,%15,%16};" ::"r"(taddr),                                                       \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),  \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),        \
      "r"(r[15])                                                                              \
      : "memory")

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Partial accumulators go through L2 only (.cg): another SM wrote them.
__device__ __forceinline__ uint4 ld_cg_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cg_v4(void* ptr, uint4 v) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void flag_release(unsigned long long* f, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long flag_acquire(const unsigned long long* f) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ void flag_clear(unsigned long long* f) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(0ull) : "memory");
}

// Waits until *f == v, then clears it for the next launch; gives up after
// `timeout_ns`, flagging the error word.
__device__ __forceinline__ bool flag_wait_bounded(unsigned long long* f, unsigned long long v,
                                                  unsigned* err_word, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (flag_acquire(f) == v) {
      flag_clear(f);
      return true;
    }
    if ((i & 15u) == 15u) {
      if (globaltimer_ns() - t0 > timeout_ns) {
        atomicOr(err_word, kErrTimeout);
        return false;
      }
      __nanosleep(256);
    }
  }
}

// ---- epilogue store of 16 consecutive fp32 accumulator columns ------------
__device__ __forceinline__ void store16(void* y, size_t idx, const uint32_t (&r)[16], bool f32) {
  if (f32) {
    float* p = static_cast<float*>(y) + idx;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(p + 4 * q) =
          make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
  } else {
    uint16_t* p = static_cast<uint16_t*>(y) + idx;
    uint32_t h[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      h[q] = pack_bf16x2_rn(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]));
    *reinterpret_cast<uint4*>(p) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(p + 8) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

__global__ void __launch_bounds__(kThreadsG, 1) agmm_kernel(const __grid_constant__ AgmmParams p) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageA;
  uint8_t* sY = sB + kStages * kStageB;  // the epilogue staging tile (1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sY + kStageY);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tmem_full = bars + 2 * kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* tmem_loaded = tmem_empty + 2;  // a partial accumulator is in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_loaded + 1);
  volatile int* aborted = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_m * p.tiles_n * p.dup;
  const int n_items = cta_items(p, num_tiles);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(tmem_loaded, 4);
    *aborted = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(tmem_slot)),
        "r"(kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (producer_index(warp) >= 0 && lane == 0) {
    // ------------------------------ TMA producers -----------------------------
    // producer i fills the stages s with s % kProducerWarps == i; all walk the
    // same sequence of k-blocks and keep the same stage/phase bookkeeping
    const int par = producer_index(warp);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed_phase[kStages];
    bool armed[kStages];
    for (int s = 0; s < kStages; ++s) armed[s] = false;
    const uint32_t tx_bytes = kStageA + (uint32_t)p.BN * BK * 2;
    for (int w = 0; w < n_items && !*aborted; ++w) {
      const Item it = cta_item(p, w);
      const int m0 = (it.tile / p.tiles_n) * BM;
      const int n0 = (it.tile % p.tiles_n) * p.BN;
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        if (stage % kProducerWarps != par) {  // the other producer's stage
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, p.err, kTimeoutNs)) {
          *aborted = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], tx_bytes);
        armed[stage] = true;
        armed_phase[stage] = phase;
        if (p.mode == kGatherB) {
          tma_load_2d(&p.tmA[0], &full[stage], sA + stage * kStageA, kb * BK, m0);
          for (int b = 0; b < p.boxes; ++b) {
            const int row = n0 + b * p.box_rows;
            const int shard = row / p.F_shard;
            tma_load_2d(&p.tmB[shard], &full[stage], sB + stage * kStageB + b * p.box_rows * 128,
                        kb * BK, row - shard * p.F_shard);
          }
        } else if (p.mode == kShardK) {
          const int r = kb / p.kb_per_rank;
          const int kx = (kb - r * p.kb_per_rank) * BK;
          tma_load_2d(&p.tmA[r], &full[stage], sA + stage * kStageA, kx, m0);
          tma_load_2d(&p.tmB[r], &full[stage], sB + stage * kStageB, kx, n0);
        } else if (p.mode == kShardKxw) {
          // x_r's k-block as in kShardK; w_r rows [kx, kx + 64), columns
          // [n0, n0 + BN) as BN / 64 slabs of 64 rows x 128 bytes
          const int r = kb / p.kb_per_rank;
          const int kx = (kb - r * p.kb_per_rank) * BK;
          tma_load_2d(&p.tmA[r], &full[stage], sA + stage * kStageA, kx, m0);
          tma_load_3d(&p.tmB[r], &full[stage], sB + stage * kStageB, kx, n0 / 64);
        } else {
          // tokens [t0, t0 + 64) of rank r; features in blocks of 64
          const int r = kb / p.kb_per_rank;
          const int t0 = (kb - r * p.kb_per_rank) * BK;
          tma_load_3d(&p.tmA[r], &full[stage], sA + stage * kStageA, t0, m0 / 64);
          tma_load_3d(&p.tmB[r], &full[stage], sB + stage * kStageB, t0, n0 / 64);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Drain: every load this thread issued has landed before the CTA exits.
    for (int s = 0; s < kStages; ++s)
      if (armed[s]) (void)mbar_wait_bounded(&full[s], armed_phase[s], p.err, kTimeoutNs);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------ MMA issuer --------------------------------
    // operand majorness: A MN-major only for the weight gradient; B also
    // for the x . w orientation (the instruction's two transpose bits)
    const bool a_mn = p.mode == kShardT;
    const bool b_mn = p.mode == kShardT || p.mode == kShardKxw;
    const uint32_t idesc =
        idesc_bf16_f32(BM, p.BN) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
    int stage = 0;
    uint32_t phase = 0;
    int last_acc = -1;
    uint32_t last_acc_phase = 0;
    uint32_t loads = 0;
    for (int w = 0; w < n_items && !*aborted; ++w) {
      const Item it = cta_item(p, w);
      const int acc = w & 1;
      const uint32_t acc_phase = (uint32_t)(w >> 1) & 1u;
      if (!mbar_wait_bounded(&tmem_empty[acc], acc_phase ^ 1u, p.err, kTimeoutNs)) {
        *aborted = 1;
        break;
      }
      if (it.load >= 0) {  // the chain continues from a partial the epilogue loaded
        if (!mbar_wait_bounded(tmem_loaded, loads & 1u, p.err, kTimeoutNs)) {
          *aborted = 1;
          break;
        }
        ++loads;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kAccCols);
      const uint32_t acc0 = it.load >= 0 ? 1u : 0u;  // first MMA: overwrite or continue
      bool ok = true;
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase, p.err, kTimeoutNs)) {
          *aborted = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * kStageA);
        const uint32_t b0 = smem_u32(sB + stage * kStageB);
        // 16 k per MMA: 32 bytes further along a K-major row, or two 8-row
        // groups (2 KiB) further on in an MN-major slab; one loop per
        // operand layout, so each issues from constant descriptor offsets
        if (a_mn) {
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(d_tmem, sw128_mnmajor_desc(a0 + 2048u * k),
                     sw128_mnmajor_desc(b0 + 2048u * k), idesc,
                     (kb > it.kb0 || k > 0) ? 1u : acc0);
        } else if (b_mn) {
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(d_tmem, sw128_kmajor_desc(a0 + 32u * k), sw128_mnmajor_desc(b0 + 2048u * k),
                     idesc, (kb > it.kb0 || k > 0) ? 1u : acc0);
        } else {
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(d_tmem, sw128_kmajor_desc(a0 + 32u * k), sw128_kmajor_desc(b0 + 32u * k),
                     idesc, (kb > it.kb0 || k > 0) ? 1u : acc0);
        }
        mma_commit(&empty[stage]);  // stage is free once these MMAs have read it
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit(&tmem_full[acc]);  // accumulator complete
      last_acc = acc;
      last_acc_phase = acc_phase;
    }
    // Drain: the last accumulator's MMAs have completed before TMEM is freed.
    if (last_acc >= 0)
      (void)mbar_wait_bounded(&tmem_full[last_acc], last_acc_phase, p.err, kTimeoutNs);
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------ epilogue ----------------------------------
    const int ew = warp - 4;  // TMEM lanes 32*ew .. 32*ew+31
    const int row = ew * 32 + lane;
    const bool leader = (ew == 0 && lane == 0);
    const bool f32 = p.y_f32 != 0;
    const uint32_t lanes = (uint32_t)(ew * 32) << 16;
    // Loads the partial accumulator that item v continues from (if any) into
    // its TMEM slot, which is free: v < 2, or item v-2's epilogue is done.
    auto load_partial = [&](int v) {
      const Item iv = cta_item(p, v);
      if (iv.load < 0) return;
      bool ok = true;
      if (leader) ok = flag_wait_bounded(&p.ws_flag[iv.load], p.nonce, p.err, kTimeoutNs);
      if (epi_any(!ok)) {
        *aborted = 1;
      } else {
        const uint32_t tb = tmem_base + lanes + (uint32_t)((v & 1) * kAccCols);
        const float* src = p.ws_part + (size_t)iv.load * BM * p.BN;
        for (int c = 0; c < p.BN; c += 16) {
          const float* q = src + ((size_t)(c / 16) * BM + row) * 16;
          uint32_t r[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 u = ld_cg_v4(q + 4 * k);
            r[4 * k] = u.x;
            r[4 * k + 1] = u.y;
            r[4 * k + 2] = u.z;
            r[4 * k + 3] = u.w;
          }
          DP_TMEM_ST_X16(tb + (uint32_t)c, r);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_loaded);
    };
    for (int v = 0; v < 2 && v < n_items; ++v) load_partial(v);
    for (int w = 0; w < n_items; ++w) {
      const Item it = cta_item(p, w);
      const int acc = w & 1;
      const uint32_t acc_phase = (uint32_t)(w >> 1) & 1u;
      const bool ok = mbar_wait_bounded(&tmem_full[acc], acc_phase, p.err, kTimeoutNs);
      if (epi_any(!ok || *aborted)) {  // all 128 epilogue threads leave together
        *aborted = 1;
        break;
      }
      tc_fence_after();
      const int m0 = (it.tile / p.tiles_n) * BM;
      const int m = m0 + row;
      const int n0 = (it.tile % p.tiles_n) * p.BN;
      const uint32_t tbase = tmem_base + lanes + (uint32_t)(acc * kAccCols);
      if (it.store >= 0) {
        // hand the fp32 accumulator on to the tile's next segment
        float* dst = p.ws_part + (size_t)it.store * BM * p.BN;
        for (int c = 0; c < p.BN; c += 16) {
          uint32_t r[16];
          DP_TMEM_LD_X16(tbase + (uint32_t)c, r);
          tmem_ld_wait();
          float* q = dst + ((size_t)(c / 16) * BM + row) * 16;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_cg_v4(q + 4 * k, make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]));
        }
        __threadfence();
        epi_bar();
        if (leader) flag_release(&p.ws_flag[it.store], p.nonce);
      } else if (p.tma_epi) {
        for (int cb = 0; cb < p.BN; cb += p.ec) {
          uint8_t* buf = sY;
          if (leader) bulk_wait_read0();  // the previous block's stores have read `buf`
          epi_bar();
          for (int q = 0; q < p.ec; q += 16) {
            uint32_t r[16];
            DP_TMEM_LD_X16(tbase + (uint32_t)(cb + q), r);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(__uint_as_float(r[e]), p.scale);
            // 128-byte swizzle: 16-byte unit u of a row sits at unit u ^ (row % 8)
            uint8_t* rowp = buf + row * 128;
            if (f32) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int u = (q / 4) + k;
                *reinterpret_cast<uint4*>(rowp + ((u ^ (row & 7)) << 4)) =
                    make_uint4(__float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]),
                               __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
              }
            } else {
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int u = (q / 8) + k;
                *reinterpret_cast<uint4*>(rowp + ((u ^ (row & 7)) << 4)) = make_uint4(
                    pack_bf16x2_rn(v[8 * k], v[8 * k + 1]), pack_bf16x2_rn(v[8 * k + 2], v[8 * k + 3]),
                    pack_bf16x2_rn(v[8 * k + 4], v[8 * k + 5]),
                    pack_bf16x2_rn(v[8 * k + 6], v[8 * k + 7]));
              }
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          epi_bar();
          if (leader) {
            int nst = 1, x = n0 + cb, y = m0, j0 = 0;
            if (p.out_mode == kOutReplicate) {
              nst = p.K / p.dup;
              j0 = it.grp * nst;
            } else if (p.out_mode == kOutRowShard) {
              j0 = m0 / p.rows_per_shard;
              y = m0 - j0 * p.rows_per_shard;
            }
            if (p.out_evict_first) {
              const uint64_t pol = l2_policy_evict_first();
              for (int j = 0; j < nst; ++j) tma_store_2d_hint(&p.tmY[j0 + j], buf, x, y, pol);
            } else {
              for (int j = 0; j < nst; ++j) tma_store_2d(&p.tmY[j0 + j], buf, x, y);
            }
            bulk_commit();
          }
        }
      } else {
        for (int col = 0; col < p.BN; col += 16) {
          uint32_t r[16];
          DP_TMEM_LD_X16(tbase + (uint32_t)col, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 16; ++q)
            r[q] = __float_as_uint(__fmul_rn(__uint_as_float(r[q]), p.scale));
          if (m < p.M) {
            if (p.out_mode == kOutOne) {
              store16(p.y[0], (size_t)m * p.F + n0 + col, r, f32);
            } else if (p.out_mode == kOutReplicate) {
              const int nc = p.K / p.dup;
              for (int j = it.grp * nc; j < (it.grp + 1) * nc; ++j)
                store16(p.y[j], (size_t)m * p.F + n0 + col, r, f32);
            } else {
              const int c = m / p.rows_per_shard;
              store16(p.y[c], (size_t)(m - c * p.rows_per_shard) * p.F + n0 + col, r, f32);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[acc]);
      if (w + 2 < n_items) load_partial(w + 2);
    }
    if (leader) bulk_wait_all();  // staged output has been written out before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---- host side -------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode != nullptr;
}

// Encoded tensor maps are cached: a map depends only on (address, shape,
// box, element type, swizzle), so repeated calls on the same buffers skip the
// host-side encoding.  Small round-robin table under a mutex.
struct MapKey {
  uintptr_t base;
  int rows, cols, box_rows, kind;  // kind 0: K-major bf16 operand; 1/2: bf16/fp32 output
  bool operator==(const MapKey& o) const {
    return base == o.base && rows == o.rows && cols == o.cols && box_rows == o.box_rows &&
           kind == o.kind;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = (uint64_t)k.base * 0x9E3779B97F4A7C15ull;
    h ^= ((uint64_t)(uint32_t)k.rows << 32 | (uint32_t)k.cols) + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    h ^= ((uint64_t)(uint32_t)k.box_rows << 8 | (uint32_t)k.kind) + (h << 6) + (h >> 2);
    return (size_t)h;
  }
};
constexpr size_t kMapCacheMax = 4096;
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

template <typename EncodeFn>
bool cached_map(CUtensorMap* map, const MapKey& key, EncodeFn encode) {
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *map = it->second;
      return true;
    }
  }
  if (!encode(map)) return false;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
  g_map_cache.emplace(key, *map);
  return true;
}

// Output map for the TMA-store epilogue: row-major [rows, cols] of bf16 or
// fp32, box [128 rows, 128 bytes], 128-byte swizzle (matching the staging tile).
bool encode_output(CUtensorMap* map, void* base, int rows, int cols, bool f32) {
  const MapKey key{reinterpret_cast<uintptr_t>(base), rows, cols, BM, f32 ? 2 : 1};
  return cached_map(map, key, [&](CUtensorMap* m) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * (f32 ? 4 : 2)};
    cuuint32_t box[2] = {(cuuint32_t)(f32 ? 32 : 64), (cuuint32_t)BM};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  });
}

// Enables the TMA-store epilogue when the tile width is a whole number of
// 128-byte output blocks and (for row shards) tiles never straddle a shard.
void setup_tma_epilogue(AgmmParams& p, void* const* ys, int nout, int rows_per_out) {
  p.ec = p.y_f32 ? 32 : 64;
  p.tma_epi = 0;
  // K copies of the output (the all-reduce form) are K times the bytes of the
  // operands and would otherwise evict them from L2 mid-kernel.
  p.out_evict_first = p.out_mode == kOutReplicate ? 1 : 0;
  if (p.BN % p.ec) return;
  if (p.out_mode == kOutRowShard && (p.rows_per_shard % BM)) return;
  for (int j = 0; j < nout; ++j)
    if (!encode_output(&p.tmY[j], ys[j], rows_per_out, p.F, p.y_f32 != 0)) return;
  p.tma_epi = 1;
}

bool encode_kmajor_bf16(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
  const MapKey key{reinterpret_cast<uintptr_t>(base), rows, cols, box_rows, 0};
  return cached_map(map, key, [&](CUtensorMap* m) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  });
}

// An MN-major operand of kShardT: the row-major [rows = T, cols] bf16 matrix
// viewed as (64 columns, T rows, cols / 64 blocks), box [64, 64 tokens,
// blocks], so one load brings `blocks` 64-column slabs of 64 tokens, each slab
// 64 rows x 128 bytes (8 KiB), 128-byte swizzled.  Needs cols % 64 == 0.
bool encode_mnmajor3_bf16(CUtensorMap* map, const void* base, int rows, int cols, int blocks) {
  const MapKey key{reinterpret_cast<uintptr_t>(base), rows, cols, blocks, 4};
  return cached_map(map, key, [&](CUtensorMap* m) {
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)BK, (cuuint32_t)blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  });
}

// Tile width along F.  A tile must never straddle a shard boundary partially:
// either it lies inside one shard (F_shard % BN == 0, one TMA box) or it is a
// whole number of shards (BN % F_shard == 0, one box per shard).
bool bn_ok(int bn, int F_shard, int K) {
  if (bn < 16 || bn > kMaxBN || bn % 16) return false;
  if (F_shard % bn == 0) return true;
  if (bn % F_shard == 0) {
    const int g = bn / F_shard;
    return K % g == 0;
  }
  return false;
}

int choose_bn(int M, int F_shard, int K, int sm_count) {
  int bn = 0;
  for (int c = kMaxBN; c >= 16; c -= 16)
    if (bn_ok(c, F_shard, K)) {
      bn = c;
      break;
    }
  if (!bn) return 0;
  const long long tiles_m = (M + BM - 1) / BM;
  // Small problems: narrower tiles give more CTAs to share the work, down to
  // 16 columns (x[128,512] . w[512,512]^T from a CUDA graph: 64 wide 6.35 us,
  // 16 wide 5.74-5.84 us per launch).
  while (tiles_m * ((long long)K * F_shard / bn) < sm_count / 2 && bn > 16 && bn % 32 == 0 &&
         bn_ok(bn / 2, F_shard, K))
    bn /= 2;
  return bn;
}

}  // namespace

namespace {

// Persistent grid: one CTA per SM (or the process-wide GEMM CTA limit).
int gemm_grid(int tiles, int sm_count) {
  int grid = tiles < sm_count ? tiles : sm_count;
  const int limit = dph::gemm_cta_limit();
  if (limit > 0 && grid > limit) grid = limit;
  return grid;
}

// The chained split of the last round for `tiles` tiles of `num_kb` k-blocks
// on `grid` CTAs: segments per tail tile (1: no split) and workspace bytes.
// Worth it when the last round is less than half full (R <= G/2): that round
// then takes 1/s of a tile instead of a whole one.  Segment j needs j whole
// tiles of its CTA before it (s <= q + 1), and segments keep >= kMinSegKb
// k-blocks.
struct SplitPlan {
  int s, q, R;
  size_t flag_bytes, bytes;
};

SplitPlan plan_split(int tiles, int grid, int num_kb, int bn) {
  SplitPlan sp{1, 0, 0, 0, 0};
  if (grid < 2) return sp;
  const int q = tiles / grid, R = tiles - q * grid;
  if (q < 1 || R == 0 || 2 * R > grid) return sp;
  int s = grid / R;
  if (s > q + 1) s = q + 1;
  if (s > kMaxSplit) s = kMaxSplit;
  while (s > 1 && num_kb / s < kMinSegKb) --s;
  if (s < 2) return sp;
  const size_t parts = (size_t)(s - 1) * (size_t)R;
  sp.s = s;
  sp.q = q;
  sp.R = R;
  sp.flag_bytes = (parts * sizeof(unsigned long long) + 255) & ~(size_t)255;
  sp.bytes = sp.flag_bytes + parts * (size_t)BM * (size_t)bn * sizeof(float);
  return sp;
}

// Flag values: distinct per launch (a graph replay reuses its launch's value,
// which is safe because every flag is cleared once it has been read).
unsigned long long next_nonce() {
  static std::atomic<unsigned long long> counter{0};
  static const unsigned long long salt =
      (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() << 20;
  unsigned long long v;
  do {
    v = salt ^ (counter.fetch_add(1) + 1);
  } while (v == 0);
  return v;
}

}  // namespace

namespace dpl {

namespace {

cudaError_t launch_params(AgmmParams& p, const dph::DeviceInfo& dev, cudaStream_t s,
                          void* ws = nullptr, size_t ws_bytes = 0) {
  if (dph::prepare_kernel(reinterpret_cast<const void*>(agmm_kernel), kThreadsG, kSmemBytes,
                          dev.device) < 1)
    return cudaErrorInvalidConfiguration;
  p.err = dev.err_word;
  const int tiles = p.tiles_m * p.tiles_n;
  // A replicate-output problem with fewer tiles than half the CTAs it may
  // use: dup CTAs share each tile, each recomputing it and storing K / dup of
  // its K copies, so the copies leave through more SMs (such a problem has no
  // part-full round to split).
  p.dup = 1;
  if (p.out_mode == kOutReplicate) {
    const int lim = dph::gemm_cta_limit();
    const int cap = lim > 0 && lim < dev.sm_count ? lim : dev.sm_count;
    while (p.dup < p.K && p.K % (2 * p.dup) == 0 && (long long)tiles * 2 * p.dup <= cap)
      p.dup *= 2;
  }
  const int grid = gemm_grid(tiles * p.dup, dev.sm_count);
  p.split_s = 1;
  if (ws && p.dup == 1) {
    const SplitPlan sp = plan_split(tiles, grid, p.num_kb, p.BN);
    if (sp.s > 1 && sp.bytes <= ws_bytes) {
      p.split_s = sp.s;
      p.split_q = sp.q;
      p.split_R = sp.R;
      p.ws_flag = static_cast<unsigned long long*>(ws);
      p.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sp.flag_bytes);
      p.nonce = next_nonce();
    }
  }
  agmm_kernel<<<grid, kThreadsG, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

bool device_ok(const dph::DeviceInfo& dev) {
  return dev.cc_major == 10 && dev.cc_minor == 3 && dev.smem_optin >= kSmemBytes && get_encoder();
}

}  // namespace

size_t allgather_matmul_workspace_bytes(int M, int D, int K, int F_shard,
                                        const dph::DeviceInfo& dev) {
  if (M < 1 || D < 1 || K < 1 || F_shard < 1) return 0;
  const int bn = choose_bn(M, F_shard, K, dev.sm_count);
  if (!bn) return 0;
  const int tiles = ((M + BM - 1) / BM) * (K * F_shard / bn);
  return plan_split(tiles, gemm_grid(tiles, dev.sm_count), (D + BK - 1) / BK, bn).bytes;
}

cudaError_t launch_allgather_matmul(const AgmmArgs& a, const dph::DeviceInfo& dev,
                                    cudaStream_t s) {
  if (!device_ok(dev)) return cudaErrorNotSupported;
  const int bn = choose_bn(a.M, a.F_shard, a.K, dev.sm_count);
  if (!bn) return cudaErrorNotSupported;

  AgmmParams p;
  memset(&p, 0, sizeof p);
  p.y[0] = a.y;
  p.M = a.M;
  p.D = a.D;
  p.F_shard = a.F_shard;
  p.F = a.K * a.F_shard;
  p.BN = bn;
  p.box_rows = bn < a.F_shard ? bn : a.F_shard;
  p.boxes = bn / p.box_rows;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = p.F / bn;
  p.num_kb = (a.D + BK - 1) / BK;
  p.y_f32 = a.y_dtype == DP_FP32 ? 1 : 0;
  p.mode = kGatherB;
  p.out_mode = kOutOne;
  p.K = a.K;
  p.scale = 1.0f;
  if (!encode_kmajor_bf16(&p.tmA[0], a.x, a.M, a.D, BM)) return cudaErrorNotSupported;
  for (int k = 0; k < a.K; ++k)
    if (!encode_kmajor_bf16(&p.tmB[k], a.w[k], a.F_shard, a.D, p.box_rows))
      return cudaErrorNotSupported;
  setup_tma_epilogue(p, p.y, 1, a.M);
  return launch_params(p, dev, s, a.workspace, a.workspace_bytes);
}

namespace {

// Tile width of the tensor-parallel GEMMs: the widest that divides F;
// narrower for small problems (0: F has no width).
int mmr_bn(int M, int F, int sm_count) {
  int bn = 0;
  for (int c = kMaxBN; c >= 16; c -= 16)
    if (F % c == 0) {
      bn = c;
      break;
    }
  if (!bn) return 0;
  const long long tiles_m = (M + BM - 1) / BM;
  while (tiles_m * (F / bn) < sm_count / 2 && bn > 64 && bn % 32 == 0) bn /= 2;
  return bn;
}

// The same for the x . w orientation, whose B tile is read as 64-column
// slabs: the widest multiple of 64 up to 256 that divides F, halved (while it
// stays a multiple of 64) for small problems (0: F % 64 != 0).
int mmr_bn_xw(int M, int F, int sm_count) {
  int bn = 0;
  for (int c = kMaxBN; c >= 64; c -= 64)
    if (F % c == 0) {
      bn = c;
      break;
    }
  if (!bn) return 0;
  const long long tiles_m = (M + BM - 1) / BM;
  while (tiles_m * (F / bn) < sm_count / 2 && bn > 64 && bn % 128 == 0) bn /= 2;
  return bn;
}

}  // namespace

size_t matmul_reduce_workspace_bytes(int K, int M, int D_shard, int F, bool w_kn,
                                     const dph::DeviceInfo& dev) {
  if (K < 1 || M < 1 || D_shard < 1 || F < 1) return 0;
  const int bn = w_kn ? mmr_bn_xw(M, F, dev.sm_count) : mmr_bn(M, F, dev.sm_count);
  if (!bn) return 0;
  const int tiles = ((M + BM - 1) / BM) * (F / bn);
  const int num_kb = K * ((D_shard + BK - 1) / BK);
  return plan_split(tiles, gemm_grid(tiles, dev.sm_count), num_kb, bn).bytes;
}

cudaError_t launch_matmul_reduce(const MmrArgs& a, const dph::DeviceInfo& dev, cudaStream_t s) {
  if (!device_ok(dev)) return cudaErrorNotSupported;
  const int bn = a.w_kn ? mmr_bn_xw(a.M, a.F, dev.sm_count) : mmr_bn(a.M, a.F, dev.sm_count);
  if (!bn) return cudaErrorNotSupported;
  const long long tiles_m = (a.M + BM - 1) / BM;

  AgmmParams p;
  memset(&p, 0, sizeof p);
  for (int k = 0; k < a.K; ++k) p.y[k] = a.y[k];
  p.M = a.M;
  p.D = a.D_shard;
  p.F = a.F;
  p.F_shard = a.F;
  p.BN = bn;
  p.box_rows = bn;
  p.boxes = 1;
  p.tiles_m = (int)tiles_m;
  p.tiles_n = a.F / bn;
  p.kb_per_rank = (a.D_shard + BK - 1) / BK;
  p.num_kb = a.K * p.kb_per_rank;
  p.y_f32 = a.y_dtype == DP_FP32 ? 1 : 0;
  p.mode = a.w_kn ? kShardKxw : kShardK;
  p.out_mode = a.scatter ? kOutRowShard : kOutReplicate;
  p.K = a.K;
  p.rows_per_shard = a.scatter ? a.M / a.K : 0;
  p.scale = a.scale;
  for (int k = 0; k < a.K; ++k) {
    if (!encode_kmajor_bf16(&p.tmA[k], a.x[k], a.M, a.D_shard, BM)) return cudaErrorNotSupported;
    const bool okb = a.w_kn ? encode_mnmajor3_bf16(&p.tmB[k], a.w[k], a.D_shard, a.F, bn / 64)
                            : encode_kmajor_bf16(&p.tmB[k], a.w[k], a.F, a.D_shard, bn);
    if (!okb) return cudaErrorNotSupported;
  }
  setup_tma_epilogue(p, p.y, a.K, a.scatter ? a.M / a.K : a.M);
  return launch_params(p, dev, s, a.workspace, a.workspace_bytes);
}

namespace {

// Tile width along D for the weight gradient: the widest multiple of 64 that
// divides D (narrower tiles measured slower here even where they fill the
// last round better: 128 x 128 tiles need 32 KiB of operands per k-block for
// half the MMA work, and intake per SM is the limit); narrower only for small
// problems so more SMs share the work.
int wgrad_bn(int F, int D, int sm_count) {
  int bn = 64;
  for (int c = kMaxBN; c >= 64; c -= 64)
    if (D % c == 0) {
      bn = c;
      break;
    }
  const long long tiles_m = (F + BM - 1) / BM;
  while (tiles_m * (D / bn) < sm_count / 2 && bn > 64 && bn % 128 == 0) bn /= 2;
  return bn;
}

}  // namespace

size_t wgrad_workspace_bytes(int K, int T, int F, int D, const dph::DeviceInfo& dev) {
  if (K < 1 || T < 1 || F < 64 || D < 64 || F % 64 || D % 64) return 0;
  const int bn = wgrad_bn(F, D, dev.sm_count);
  const int tiles = ((F + BM - 1) / BM) * (D / bn);
  const int num_kb = K * ((T + BK - 1) / BK);
  return plan_split(tiles, gemm_grid(tiles, dev.sm_count), num_kb, bn).bytes;
}

cudaError_t launch_wgrad_reduce_scatter(const WgradArgs& a, const dph::DeviceInfo& dev,
                                        cudaStream_t s) {
  if (!device_ok(dev)) return cudaErrorNotSupported;
  if (a.F % 64 != 0 || a.D % 64 != 0) return cudaErrorNotSupported;
  const int bn = wgrad_bn(a.F, a.D, dev.sm_count);
  const long long tiles_m = (a.F + BM - 1) / BM;

  AgmmParams p;
  memset(&p, 0, sizeof p);
  for (int k = 0; k < a.K; ++k) p.y[k] = a.y[k];
  p.M = a.F;  // the product's rows are the output features
  p.D = a.T;
  p.F = a.D;  // ... and its columns the input features
  p.F_shard = a.D;
  p.BN = bn;
  p.box_rows = bn;
  p.boxes = 1;
  p.tiles_m = (int)tiles_m;
  p.tiles_n = a.D / bn;
  p.kb_per_rank = (a.T + BK - 1) / BK;
  p.num_kb = a.K * p.kb_per_rank;
  p.y_f32 = a.y_dtype == DP_FP32 ? 1 : 0;
  p.mode = kShardT;
  p.out_mode = kOutRowShard;
  p.K = a.K;
  p.rows_per_shard = a.F / a.K;
  p.scale = a.scale;
  for (int k = 0; k < a.K; ++k) {
    if (!encode_mnmajor3_bf16(&p.tmA[k], a.dy[k], a.T, a.F, BM / 64) ||
        !encode_mnmajor3_bf16(&p.tmB[k], a.x[k], a.T, a.D, bn / 64))
      return cudaErrorNotSupported;
  }
  setup_tma_epilogue(p, p.y, a.K, a.F / a.K);
  return launch_params(p, dev, s, a.workspace, a.workspace_bytes);
}

}  // namespace dpl
