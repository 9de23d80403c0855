/*
 * ring_oracle.c -- the CPU oracle for the data-parallel gradient/parameter
 * collective path.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code,
 * header, table or helper with the CUDA library; nothing in the product
 * path calls it.
 *
 * It is deliberately plain and slow: scalar loops, fp32 arithmetic exactly
 * as written (build with -O2 -ffp-contract=off, no fast-math), fp64 for the
 * GEMM reference.  Each routine cites the passage it follows.
 *
 * Sources (web pages):
 *  [CMU] "CMU 11-868 L14-L15: Distributed Training and Data Parallelism, and
 *        Where Gradient Sync Costs Come From", section "Ring AllReduce:
 *        ReduceScatter, then AllGather" (the 4-worker a0..d3 walk: every
 *        worker splits its gradient into K chunks; at each of K-1 steps every
 *        worker sends one chunk to the next worker, which adds it to its own
 *        matching chunk; then K-1 copy steps pass the finished chunks on),
 *        section "NCCL's five building blocks" (AllReduce = ReduceScatter +
 *        AllGather), section "Intuition: data parallelism has only one thing
 *        to synchronize" (step 3: workers compute the average gradient).
 *  [SHARD] "Sharding and Parallelism" (How to Scale Your Model on AMD,
 *        ch. 5), section "Real HLO before and after partitioning" (FSDP
 *        fixture: all-gather w[64,512] shards to w[512,512], then the local
 *        dot) and section "FSDP and ZeRO" (the forward pass gathers W before
 *        the dot).
 *  [ODC] "Using ODC to Accelerate AMD SFT Training", sections "From
 *        Per-iteration to Per-minibatch Synchronization" (microbatch
 *        gradients accumulate locally, one settle per minibatch),
 *        "odc_pad vs odc_nopad" (Figure 5: padding buckets contribute no
 *        valid gradient) and "Discussion: Settle Does Not Yet Overlap with
 *        Backward" (a cross-iteration pipeline settles the previous
 *        microbatch group beside this group's backward).
 *
 * Readings fixed where the pages are silent:
 *  - At step s rank r sends chunk (r-s-1) mod K to rank (r+1) mod K, so the
 *    reduced chunk c ends on rank c and is folded in the order
 *    x_{c+1}, x_{c+2}, ..., x_{c} (indices mod K).
 *  - The fold is fp32 throughout; bf16 inputs are widened exactly (bf16 is
 *    the upper half of a binary32).  The average is one fp32 multiply by
 *    `scale` after the fold, then one rounding to the output type.
 *  - bf16 output rounding is round-to-nearest, ties-to-even; NaN stays a
 *    quiet NaN.
 *  - For the all-reduce, C = ceil(N/K); trailing chunks may be short or
 *    empty.  Reduce-scatter and all-gather require N % K == 0.
 *  - A microbatch accumulator starts at +0; a padding bucket adds +0; a
 *    rank's microbatches are added in ascending order j = 0, 1, ...
 *  - Pipelined settle: each microbatch group (an index range of j shared by
 *    the ranks) is settled by the ring reduce-scatter and added to the
 *    owner's +0-seeded fp32 accumulator in group order; the average and the
 *    cast come once, after the last group.
 *
 * Mutations: oracle_set_mutation() plants a known mistake so that the test
 * suite can show its pins catch it.  0 (the default) is the oracle proper.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_ENOMEM = 2, ORC_EMISMATCH = 3 };

/* Planted mistakes, for the tests that check the pins catch them. */
enum {
  MUT_NONE = 0,
  MUT_REVERSED_RING = 1,   /* send to rank r-1 instead of r+1            */
  MUT_START_AT_OWNER = 2,  /* fold chunk c starting at rank c            */
  MUT_DROP_SCALE = 3,      /* forget the average                         */
  MUT_TRUNCATE_CAST = 4,   /* bf16 cast truncates instead of rounding    */
  MUT_SKIP_LAST_STEP = 5,  /* run only K-2 reduce-scatter steps          */
  MUT_GEMM_TRANSPOSE = 6,  /* y = x . w instead of x . w^T (square only) */
  MUT_PAD_NOT_ZERO = 7,    /* a padding bucket adds 2^-24, not +0        */
  MUT_PSUM_SKIP_RANK = 8,  /* the psum leaves out the last rank          */
  MUT_ODC_SETTLE_PER_MB = 9,   /* one settle per microbatch index, summed  */
  MUT_ODC_FLAT_FOLD = 10,      /* one fold over all microbatches, ring order */
  MUT_ODC_REVERSED_MB = 11,    /* a rank's microbatches in descending order */
  MUT_ODC_PAIRWISE_MB = 12,    /* a rank's microbatches summed pairwise     */
  MUT_PIPE_CARRY_IN_FOLD = 13, /* owner's running sum seeds the group fold  */
  MUT_PIPE_REVERSED_GROUPS = 14, /* settled groups added last to first      */
  MUT_PIPE_SCALE_PER_GROUP = 15, /* the average applied to every group      */
};
static int g_mutation = MUT_NONE;

int oracle_set_mutation(int m) { int old = g_mutation; g_mutation = m; return old; }

/* ---------------------------------------------------------------------- */
/* bf16 <-> fp32 from the IEEE-754 binary32 bit layout.                     */
/* ---------------------------------------------------------------------- */

/* bf16 holds the sign, the 8 exponent bits and the top 7 fraction bits of a
 * binary32, so widening is exact: place the 16 bits in the upper half. */
static float bf16_widen(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a binary32 to the nearest bf16, ties to even.  Within one binade the
 * encoding is monotone in magnitude, and stepping past the top of a binade
 * lands on the next binade's first value (or infinity), so the two
 * candidates are the truncation `lo` and `lo + one bf16 ulp`; the 16 dropped
 * bits say which is nearer. */
static uint16_t bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u); /* NaN: keep sign/payload top, make it quiet */
  uint32_t lo = u >> 16;
  uint32_t dropped = u & 0xffffu;
  if (g_mutation == MUT_TRUNCATE_CAST) return (uint16_t)lo;
  if (dropped > 0x8000u) return (uint16_t)(lo + 1u);
  if (dropped < 0x8000u) return (uint16_t)lo;
  return (uint16_t)((lo & 1u) ? lo + 1u : lo); /* exact tie: pick the even one */
}

/* Exposed so the tests can pin the cast against an independent library. */
uint16_t oracle_bf16_round(float f) { return bf16_round(f); }
float oracle_bf16_widen(uint16_t h) { return bf16_widen(h); }

static float load_elem(const void* p, size_t i, int dtype) {
  if (dtype == ORC_F32) return ((const float*)p)[i];
  return bf16_widen(((const uint16_t*)p)[i]);
}

static void store_elem(void* p, size_t i, int dtype, float v) {
  if (dtype == ORC_F32) ((float*)p)[i] = v;
  else ((uint16_t*)p)[i] = bf16_round(v);
}

static size_t elem_size(int dtype) { return dtype == ORC_F32 ? 4u : 2u; }

static int mod(int a, int k) { int r = a % k; return r < 0 ? r + k : r; }

/* Chunk c of an N-element buffer split into K chunks of C = ceil(N/K)
 * elements ([CMU] "each worker splits its gradient into K chunks"). */
static void chunk_bounds(size_t N, int K, int c, size_t* lo, size_t* hi) {
  size_t C = (N + (size_t)K - 1) / (size_t)K;
  size_t a = (size_t)c * C, b = a + C;
  if (a > N) a = N;
  if (b > N) b = N;
  *lo = a;
  *hi = b;
}

/* ---------------------------------------------------------------------- */
/* (i) Step simulator: the ring walk of [CMU] played out between per-rank   */
/* arrays, one step at a time.                                              */
/* ---------------------------------------------------------------------- */

/* Reduce-scatter phase on fp32 working copies work[r*N .. r*N+N).
 * At step s = 0..K-2 every rank r sends its current chunk (r-s-1) mod K to
 * the next rank; the receiver adds it to its own matching chunk.  All sends
 * of a step happen "at once": the messages are copied out first. */
static int sim_reduce_scatter(float* work, int K, size_t N, int skip_rank, int skip_step) {
  if (K <= 1 || N == 0) return ORC_OK;
  size_t C = (N + (size_t)K - 1) / (size_t)K;
  float* msg = (float*)malloc((size_t)K * C * sizeof(float));
  if (!msg) return ORC_ENOMEM;
  int steps = K - 1;
  if (g_mutation == MUT_SKIP_LAST_STEP) steps = K - 2;
  for (int s = 0; s < steps; ++s) {
    /* send: rank r puts chunk (r-s-1) mod K on the wire */
    for (int r = 0; r < K; ++r) {
      int c = mod(r - s - 1, K);
      if (g_mutation == MUT_REVERSED_RING) c = mod(r + s + 1, K);
      if (g_mutation == MUT_START_AT_OWNER) c = mod(r - s, K);
      size_t lo, hi;
      chunk_bounds(N, K, c, &lo, &hi);
      for (size_t e = lo; e < hi; ++e) msg[(size_t)r * C + (e - lo)] = work[(size_t)r * N + e];
    }
    /* A rank that skips this step never sends: its successor's receive would
     * wait forever in a real ring; here the missing message is an error. */
    if (s == skip_step && skip_rank >= 0 && skip_rank < K) {
      free(msg);
      return ORC_EMISMATCH;
    }
    /* receive: the next rank adds the message to its own copy of that chunk */
    for (int r = 0; r < K; ++r) {
      int c = mod(r - s - 1, K);
      int q = mod(r + 1, K);
      if (g_mutation == MUT_REVERSED_RING) { c = mod(r + s + 1, K); q = mod(r - 1, K); }
      if (g_mutation == MUT_START_AT_OWNER) c = mod(r - s, K);
      size_t lo, hi;
      chunk_bounds(N, K, c, &lo, &hi);
      for (size_t e = lo; e < hi; ++e) {
        float own = work[(size_t)q * N + e];
        float incoming = msg[(size_t)r * C + (e - lo)];
        work[(size_t)q * N + e] = own + incoming;
      }
    }
  }
  free(msg);
  return ORC_OK;
}

/* The rank that holds the finished chunk c after the reduce-scatter phase. */
static int owner_of_chunk(int c, int K) {
  if (g_mutation == MUT_REVERSED_RING) return mod(c, K);
  if (g_mutation == MUT_START_AT_OWNER) return mod(c - 1, K);
  return c;
}

/* All-gather phase on per-rank typed buffers bufs[r] (N elements each, esz
 * bytes per element), where rank r already holds finished chunk r.
 * At step s = 0..K-2 rank r sends chunk (r-s) mod K to the next rank, which
 * stores it ([CMU] "another K-1 steps pass the finished chunks to
 * everyone"). */
static int sim_all_gather(unsigned char** bufs, int K, size_t N, size_t esz) {
  if (K <= 1 || N == 0) return ORC_OK;
  size_t C = (N + (size_t)K - 1) / (size_t)K;
  unsigned char* msg = (unsigned char*)malloc((size_t)K * C * esz);
  if (!msg) return ORC_ENOMEM;
  for (int s = 0; s < K - 1; ++s) {
    for (int r = 0; r < K; ++r) {
      int c = mod(r - s, K);
      size_t lo, hi;
      chunk_bounds(N, K, c, &lo, &hi);
      memcpy(msg + (size_t)r * C * esz, bufs[r] + lo * esz, (hi - lo) * esz);
    }
    for (int r = 0; r < K; ++r) {
      int c = mod(r - s, K);
      int q = mod(r + 1, K);
      size_t lo, hi;
      chunk_bounds(N, K, c, &lo, &hi);
      memcpy(bufs[q] + lo * esz, msg + (size_t)r * C * esz, (hi - lo) * esz);
    }
  }
  free(msg);
  return ORC_OK;
}

/* Copy the K input buffers into fp32 working arrays (exact widening). */
static float* widen_inputs(const void* const* bufs, int K, size_t N, int in_dtype) {
  float* work = (float*)malloc((size_t)K * (N ? N : 1) * sizeof(float));
  if (!work) return NULL;
  for (int r = 0; r < K; ++r)
    for (size_t e = 0; e < N; ++e) work[(size_t)r * N + e] = load_elem(bufs[r], e, in_dtype);
  return work;
}

/* The average ([CMU] DP step 3), applied once to the fp32 fold. */
static float apply_scale(float folded, float scale) {
  if (g_mutation == MUT_DROP_SCALE) return folded;
  return folded * scale;
}

static int check_common(const void* const* bufs, int K, int dt) {
  if (!bufs || K < 1) return ORC_EINVAL;
  if (dt != ORC_F32 && dt != ORC_BF16) return ORC_EINVAL;
  for (int r = 0; r < K; ++r)
    if (!bufs[r]) return ORC_EINVAL;
  return ORC_OK;
}

/* Ring reduce-scatter by simulation.  out_f32 / out_bf16: K shard pointers of
 * N/K elements each, either array may be NULL (not both).  Shard c is the
 * chunk rank c holds after the reduce-scatter phase, scaled and cast. */
/* The same walk with one rank skipping one step of the reduce-scatter phase
 * (the failure the ODC page describes in "odc_pad vs odc_nopad": collectives
 * need every rank to make the same calls, and a mismatch hangs the group).
 * Returns ORC_EMISMATCH instead of waiting; skip_rank < 0 disables it. */
int oracle_reduce_scatter_sim_skip(const void* const* bufs, int K, size_t N, int in_dtype,
                                   float scale, float* const* out_f32,
                                   uint16_t* const* out_bf16, int skip_rank, int skip_step) {
  int st = check_common(bufs, K, in_dtype);
  if (st) return st;
  if (N % (size_t)K) return ORC_EINVAL;
  if (!out_f32 && !out_bf16) return ORC_EINVAL;
  if (N == 0) return ORC_OK;
  float* work = widen_inputs(bufs, K, N, in_dtype);
  if (!work) return ORC_ENOMEM;
  st = sim_reduce_scatter(work, K, N, skip_rank, skip_step);
  if (st) { free(work); return st; }
  size_t C = N / (size_t)K;
  for (int c = 0; c < K; ++c) {
    int q = owner_of_chunk(c, K);
    for (size_t i = 0; i < C; ++i) {
      float v = apply_scale(work[(size_t)q * N + (size_t)c * C + i], scale);
      if (out_f32) out_f32[c][i] = v;
      if (out_bf16) out_bf16[c][i] = bf16_round(v);
    }
  }
  free(work);
  return ORC_OK;
}

int oracle_reduce_scatter_sim(const void* const* bufs, int K, size_t N, int in_dtype,
                              float scale, float* const* out_f32, uint16_t* const* out_bf16) {
  return oracle_reduce_scatter_sim_skip(bufs, K, N, in_dtype, scale, out_f32, out_bf16, -1, -1);
}

/* Ring all-gather by simulation: shards[c] (C elements each, dtype) end up
 * concatenated in every out[r] (K*C elements). */
int oracle_all_gather_sim(const void* const* shards, int K, size_t C, int dtype, void* const* out) {
  int st = check_common(shards, K, dtype);
  if (st) return st;
  if (!out) return ORC_EINVAL;
  for (int r = 0; r < K; ++r)
    if (!out[r]) return ORC_EINVAL;
  size_t esz = elem_size(dtype), N = (size_t)K * C;
  if (N == 0) return ORC_OK;
  /* start: rank r holds only its own finished chunk r */
  for (int r = 0; r < K; ++r) memcpy((unsigned char*)out[r] + (size_t)r * C * esz, shards[r], C * esz);
  return sim_all_gather((unsigned char**)out, K, N, esz);
}

/* Ring all-reduce by simulation: the reduce-scatter phase, the average and
 * cast on each owner, then the all-gather phase.  Inputs bufs[r] (N elements
 * of dtype); outputs out[r] (N elements of the same dtype).  Any N >= 0. */
int oracle_all_reduce_sim(const void* const* bufs, int K, size_t N, int dtype, float scale,
                          void* const* out) {
  int st = check_common(bufs, K, dtype);
  if (st) return st;
  if (!out) return ORC_EINVAL;
  for (int r = 0; r < K; ++r)
    if (!out[r]) return ORC_EINVAL;
  if (N == 0) return ORC_OK;
  float* work = widen_inputs(bufs, K, N, dtype);
  if (!work) return ORC_ENOMEM;
  st = sim_reduce_scatter(work, K, N, -1, -1);
  if (st) { free(work); return st; }
  for (int c = 0; c < K; ++c) {
    int q = owner_of_chunk(c, K);
    size_t lo, hi;
    chunk_bounds(N, K, c, &lo, &hi);
    /* the owner writes its finished, averaged, cast chunk into its own buffer */
    for (size_t e = lo; e < hi; ++e)
      store_elem(out[c], e, dtype, apply_scale(work[(size_t)q * N + e], scale));
  }
  free(work);
  return sim_all_gather((unsigned char**)out, K, N, elem_size(dtype));
}

/* ---------------------------------------------------------------------- */
/* (ii) Closed form: the same result written as a fold per element.         */
/* shard_c[i] = cast(scale * (((x_{c+1} + x_{c+2}) + ...) + x_{c})),        */
/* indices mod K, starting from the first term (no zero seed).              */
/* ---------------------------------------------------------------------- */
int oracle_reduce_scatter_fold(const void* const* bufs, int K, size_t N, int in_dtype,
                               float scale, float* const* out_f32, uint16_t* const* out_bf16) {
  int st = check_common(bufs, K, in_dtype);
  if (st) return st;
  if (N % (size_t)K) return ORC_EINVAL;
  if (!out_f32 && !out_bf16) return ORC_EINVAL;
  size_t C = N / (size_t)K;
  for (int c = 0; c < K; ++c) {
    for (size_t i = 0; i < C; ++i) {
      size_t e = (size_t)c * C + i;
      float acc = load_elem(bufs[mod(c + 1, K)], e, in_dtype);
      for (int j = 2; j <= K; ++j) acc = acc + load_elem(bufs[mod(c + j, K)], e, in_dtype);
      float v = apply_scale(acc, scale);
      if (out_f32) out_f32[c][i] = v;
      if (out_bf16) out_bf16[c][i] = bf16_round(v);
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* (iii) FSDP forward: all-gather the weight shards, then the local dot.    */
/* [SHARD] "Real HLO before and after partitioning": w_k[F_shard, D] row    */
/* shards gather to w[K*F_shard, D]; y = x . w^T, here in fp64 from the     */
/* exact bf16 values.                                                       */
/* ---------------------------------------------------------------------- */

/* Gather the row shards into one [K*F_shard, D] bf16 matrix (a plain copy). */
static uint16_t* gather_weight(const uint16_t* const* w_shards, int K, int F_shard, int D) {
  size_t F = (size_t)K * (size_t)F_shard;
  uint16_t* w = (uint16_t*)malloc((F ? F : 1) * (size_t)(D ? D : 1) * sizeof(uint16_t));
  if (!w) return NULL;
  for (int k = 0; k < K; ++k)
    memcpy(w + (size_t)k * F_shard * D, w_shards[k], (size_t)F_shard * D * sizeof(uint16_t));
  return w;
}

/* y[m, f] = sum_d x[m, d] * w[f, d] in fp64, for all m < M, f < K*F_shard. */
int oracle_allgather_matmul_f64(const uint16_t* x, int M, int D, const uint16_t* const* w_shards,
                                int K, int F_shard, double* y) {
  if (!x || !w_shards || !y || M < 0 || D < 0 || K < 1 || F_shard < 0) return ORC_EINVAL;
  for (int k = 0; k < K; ++k)
    if (!w_shards[k]) return ORC_EINVAL;
  size_t F = (size_t)K * (size_t)F_shard;
  if (g_mutation == MUT_GEMM_TRANSPOSE && F != (size_t)D) return ORC_EINVAL;
  uint16_t* w = gather_weight(w_shards, K, F_shard, D);
  if (!w) return ORC_ENOMEM;
  for (int m = 0; m < M; ++m) {
    for (size_t f = 0; f < F; ++f) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) {
        double a = (double)bf16_widen(x[(size_t)m * D + d]);
        double b;
        if (g_mutation == MUT_GEMM_TRANSPOSE)
          b = (double)bf16_widen(w[(size_t)d * F + f]);
        else
          b = (double)bf16_widen(w[f * (size_t)D + d]);
        acc += a * b;
      }
      y[(size_t)m * F + f] = acc;
    }
  }
  free(w);
  return ORC_OK;
}

/* The same dot for a list of (m, f) output positions only, for checking a
 * large product on a sample.  No gathered copy is made: row f of the gathered
 * weight is row (f mod F_shard) of shard (f / F_shard). */
int oracle_allgather_matmul_f64_sampled(const uint16_t* x, int M, int D,
                                        const uint16_t* const* w_shards, int K, int F_shard,
                                        const int64_t* ms, const int64_t* fs, int64_t count,
                                        double* out) {
  if (!x || !w_shards || !ms || !fs || !out || K < 1 || F_shard < 1) return ORC_EINVAL;
  int64_t F = (int64_t)K * F_shard;
  for (int64_t t = 0; t < count; ++t) {
    int64_t m = ms[t], f = fs[t];
    if (m < 0 || m >= M || f < 0 || f >= F) return ORC_EINVAL;
    const uint16_t* wrow = w_shards[f / F_shard] + (size_t)(f % F_shard) * D;
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += (double)bf16_widen(x[(size_t)m * D + d]) * (double)bf16_widen(wrow[d]);
    out[t] = acc;
  }
  return ORC_OK;
}

/* Tensor-parallel partial dots summed over the ranks ([SHARD] "Real HLO
 * before and after partitioning", TP-style fixture: the contracting dimension
 * is split over the ranks, each rank computes a partial dot, an all-reduce
 * sums the partials).  Rank r holds x_r [M, Ds] and w_r [F, Ds] (weight in
 * the [out, in] layout); y[m, f] = scale * sum_r partial_r[m, f] with
 * partial_r[m, f] = sum_d x_r[m, d] * w_r[f, d], all in fp64, ranks summed in
 * ascending order.  Only the (m, f) positions listed are computed. */
int oracle_matmul_psum_f64_sampled(const uint16_t* const* x_shards,
                                   const uint16_t* const* w_shards, int K, int M, int Ds, int F,
                                   double scale, const int64_t* ms, const int64_t* fs,
                                   int64_t count, double* out) {
  if (!x_shards || !w_shards || !ms || !fs || !out || K < 1 || Ds < 0) return ORC_EINVAL;
  for (int r = 0; r < K; ++r)
    if (!x_shards[r] || !w_shards[r]) return ORC_EINVAL;
  for (int64_t t = 0; t < count; ++t) {
    int64_t m = ms[t], f = fs[t];
    if (m < 0 || m >= M || f < 0 || f >= F) return ORC_EINVAL;
    double total = 0.0;
    for (int r = 0; r < K; ++r) {
      if (g_mutation == MUT_PSUM_SKIP_RANK && r == K - 1 && K > 1) break;
      double partial = 0.0;
      for (int d = 0; d < Ds; ++d)
        partial += (double)bf16_widen(x_shards[r][(size_t)m * Ds + d]) *
                   (double)bf16_widen(w_shards[r][(size_t)f * Ds + d]);
      total += partial;
    }
    out[t] = scale * total;
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* (iv) Variable-length microbatch step ([ODC]).                            */
/* ---------------------------------------------------------------------- */

/* One microbatch into one rank's fp32 accumulator:
 * acc = (first ? +0 : acc) + widen(grad); grad == NULL is a padding bucket,
 * whose gradient is +0 ([ODC] Figure 5: "contribute no valid gradient"). */
int oracle_accumulate(float* acc, const void* grad, size_t N, int grad_dtype, int first) {
  if (!acc) return ORC_EINVAL;
  if (grad_dtype != ORC_F32 && grad_dtype != ORC_BF16) return ORC_EINVAL;
  for (size_t e = 0; e < N; ++e) {
    float g = grad ? load_elem(grad, e, grad_dtype) : 0.0f;
    if (!grad && g_mutation == MUT_PAD_NOT_ZERO) g = 5.9604645e-08f; /* 2^-24 */
    float base = first ? 0.0f : acc[e];
    acc[e] = base + g;
  }
  return ORC_OK;
}

/* One rank's microbatches j = lo .. hi-1 (hi <= m_r) summed into a +0-seeded
 * fp32 accumulator in ascending order ([ODC] "From Per-iteration to
 * Per-minibatch Synchronization": gradients accumulate locally).  row is the
 * rank's row of the K x Mmax gradient table; NULL entries are padding. */
static int rank_accumulate(float* a, const void* const* row, int lo, int hi, size_t N,
                           int grad_dtype) {
  for (size_t e = 0; e < N; ++e) a[e] = 0.0f; /* +0 */
  if (g_mutation == MUT_ODC_REVERSED_MB) {
    for (int j = hi - 1; j >= lo; --j) {
      int st = oracle_accumulate(a, row[j], N, grad_dtype, 0);
      if (st) return st;
    }
    return ORC_OK;
  }
  if (g_mutation == MUT_ODC_PAIRWISE_MB && hi - lo > 1) {
    /* planted mistake: halves summed separately, then added */
    int mid = lo + (hi - lo + 1) / 2;
    float* b = (float*)malloc((N ? N : 1) * sizeof(float));
    if (!b) return ORC_ENOMEM;
    int st = rank_accumulate(a, row, lo, mid, N, grad_dtype);
    if (!st) st = rank_accumulate(b, row, mid, hi, N, grad_dtype);
    for (size_t e = 0; !st && e < N; ++e) a[e] = a[e] + b[e];
    free(b);
    return st;
  }
  for (int j = lo; j < hi; ++j) {
    int st = oracle_accumulate(a, row[j], N, grad_dtype, 0);
    if (st) return st;
  }
  return ORC_OK;
}

/* Planted mistake MUT_ODC_SETTLE_PER_MB: a ring settle for every microbatch
 * index j (ranks without a j-th microbatch give +0), the settled chunks
 * summed over j, then the average. */
static int odc_settle_per_microbatch(const void* const* grads, const int* m, int K, int Mmax,
                                     size_t N, int grad_dtype, float scale,
                                     float* const* out_f32, uint16_t* const* out_bf16) {
  size_t C = N / (size_t)K;
  float* acc = (float*)malloc((size_t)K * (N ? N : 1) * sizeof(float));
  float* tot = (float*)calloc((size_t)K * (C ? C : 1), sizeof(float));
  float* s32 = (float*)malloc((size_t)K * (C ? C : 1) * sizeof(float));
  const void** ptrs = (const void**)malloc((size_t)K * sizeof(void*));
  float** sp = (float**)malloc((size_t)K * sizeof(float*));
  int st = (acc && tot && s32 && ptrs && sp) ? ORC_OK : ORC_ENOMEM;
  for (int j = 0; !st && j < Mmax; ++j) {
    for (int r = 0; r < K; ++r) {
      const void* g = j < m[r] ? grads[(size_t)r * Mmax + j] : NULL;
      float* a = acc + (size_t)r * N;
      for (size_t e = 0; e < N; ++e) a[e] = g ? load_elem(g, e, grad_dtype) : 0.0f;
      ptrs[r] = a;
      sp[r] = s32 + (size_t)r * C;
    }
    st = oracle_reduce_scatter_sim(ptrs, K, N, ORC_F32, 1.0f, sp, NULL);
    for (size_t i = 0; !st && i < (size_t)K * C; ++i) tot[i] = tot[i] + s32[i];
  }
  for (int c = 0; !st && c < K; ++c)
    for (size_t i = 0; i < C; ++i) {
      float v = apply_scale(tot[(size_t)c * C + i], scale);
      if (out_f32) out_f32[c][i] = v;
      if (out_bf16) out_bf16[c][i] = bf16_round(v);
    }
  free(acc); free(tot); free(s32); free(ptrs); free(sp);
  return st;
}

/* Planted mistake MUT_ODC_FLAT_FOLD: chunk c folded left to right over the
 * ring-ordered list of every microbatch (rank c+1's in ascending j, then
 * rank c+2's, ..., rank c's), starting from the first term. */
static int odc_flat_fold(const void* const* grads, const int* m, int K, int Mmax, size_t N,
                         int grad_dtype, float scale, float* const* out_f32,
                         uint16_t* const* out_bf16) {
  size_t C = N / (size_t)K;
  for (int c = 0; c < K; ++c)
    for (size_t i = 0; i < C; ++i) {
      size_t e = (size_t)c * C + i;
      float acc = 0.0f;
      int started = 0;
      for (int q = 1; q <= K; ++q) {
        int r = mod(c + q, K);
        for (int j = 0; j < m[r]; ++j) {
          const void* g = grads[(size_t)r * Mmax + j];
          float v = g ? load_elem(g, e, grad_dtype) : 0.0f;
          acc = started ? acc + v : v;
          started = 1;
        }
      }
      float v = apply_scale(acc, scale);
      if (out_f32) out_f32[c][i] = v;
      if (out_bf16) out_bf16[c][i] = bf16_round(v);
    }
  return ORC_OK;
}

static int odc_check(const void* const* grads, const int* m, int K, int Mmax, size_t N) {
  if (!grads || !m || K < 1 || Mmax < 0) return ORC_EINVAL;
  if (N % (size_t)K) return ORC_EINVAL;
  for (int r = 0; r < K; ++r)
    if (m[r] < 0 || m[r] > Mmax) return ORC_EINVAL;
  return ORC_OK;
}

/* One layer of the step: each rank r runs its m[r] microbatches in order
 * j = 0..m[r]-1 into an accumulator that starts at +0; then one ring
 * reduce-scatter (the settle) over the K fp32 accumulators, the average and
 * the casts.  grads is a K x Mmax table, row-major by rank; grads[r*Mmax+j]
 * may be NULL (a padding bucket).  m[r] <= Mmax. */
int oracle_odc_layer(const void* const* grads, const int* m, int K, int Mmax, size_t N,
                     int grad_dtype, float scale, float* const* out_f32,
                     uint16_t* const* out_bf16) {
  int st = odc_check(grads, m, K, Mmax, N);
  if (st) return st;
  if (g_mutation == MUT_ODC_SETTLE_PER_MB)
    return odc_settle_per_microbatch(grads, m, K, Mmax, N, grad_dtype, scale, out_f32, out_bf16);
  if (g_mutation == MUT_ODC_FLAT_FOLD)
    return odc_flat_fold(grads, m, K, Mmax, N, grad_dtype, scale, out_f32, out_bf16);
  float* acc = (float*)malloc((size_t)K * (N ? N : 1) * sizeof(float));
  if (!acc) return ORC_ENOMEM;
  for (int r = 0; r < K; ++r) {
    st = rank_accumulate(acc + (size_t)r * N, grads + (size_t)r * Mmax, 0, m[r], N, grad_dtype);
    if (st) { free(acc); return st; }
  }
  const void** ptrs = (const void**)malloc((size_t)K * sizeof(void*));
  if (!ptrs) { free(acc); return ORC_ENOMEM; }
  for (int r = 0; r < K; ++r) ptrs[r] = acc + (size_t)r * N;
  st = oracle_reduce_scatter_sim(ptrs, K, N, ORC_F32, scale, out_f32, out_bf16);
  free(ptrs);
  free(acc);
  return st;
}

/* Cross-iteration settle pipeline ([ODC] "Discussion: Settle Does Not Yet
 * Overlap with Backward": the settle of the previous microbatch group runs
 * beside this group's backward compute, joined once per minibatch).
 * Groups are the index ranges [bounds[g], bounds[g+1]) of j, g = 0..G-1,
 * shared by all ranks (bounds non-decreasing from 0, bounds[G] >= every
 * m[r]).  For each group in order: every rank sums its microbatches of the
 * group into a +0-seeded accumulator (ascending j); the K accumulators are
 * settled by the ring reduce-scatter (no average yet); the owner of chunk c
 * adds the settled chunk to its own fp32 accumulator, which starts at +0.
 * After the last group the owners' accumulators are averaged and cast once.
 * With one group this is oracle_odc_layer. */
int oracle_odc_pipelined(const void* const* grads, const int* m, int K, int Mmax, size_t N,
                         int grad_dtype, const int* bounds, int G, float scale,
                         float* const* out_f32, uint16_t* const* out_bf16) {
  int st = odc_check(grads, m, K, Mmax, N);
  if (st) return st;
  if (!bounds || G < 1 || bounds[0] != 0) return ORC_EINVAL;
  for (int g = 0; g < G; ++g)
    if (bounds[g + 1] < bounds[g]) return ORC_EINVAL;
  for (int r = 0; r < K; ++r)
    if (m[r] > bounds[G]) return ORC_EINVAL;
  size_t C = N / (size_t)K;
  float* acc = (float*)malloc((size_t)K * (N ? N : 1) * sizeof(float));
  float* owner = (float*)malloc((size_t)K * (C ? C : 1) * sizeof(float));
  float* settled = (float*)malloc((size_t)G * K * (C ? C : 1) * sizeof(float));
  const void** ptrs = (const void**)malloc((size_t)K * sizeof(void*));
  float** sp = (float**)malloc((size_t)K * sizeof(float*));
  if (!acc || !owner || !settled || !ptrs || !sp) {
    free(acc); free(owner); free(settled); free(ptrs); free(sp);
    return ORC_ENOMEM;
  }
  for (size_t i = 0; i < (size_t)K * C; ++i) owner[i] = 0.0f; /* +0 */
  for (int g = 0; !st && g < G; ++g) {
    float* sg = settled + (size_t)g * K * C;
    for (int r = 0; !st && r < K; ++r) {
      int lo = bounds[g], hi = bounds[g + 1] < m[r] ? bounds[g + 1] : m[r];
      if (hi < lo) hi = lo;
      st = rank_accumulate(acc + (size_t)r * N, grads + (size_t)r * Mmax, lo, hi, N, grad_dtype);
      ptrs[r] = acc + (size_t)r * N;
      sp[r] = sg + (size_t)r * C;
    }
    if (st) break;
    if (g_mutation == MUT_PIPE_CARRY_IN_FOLD) {
      /* planted mistake: the owner's value opens the fold of the group */
      for (int c = 0; c < K; ++c)
        for (size_t i = 0; i < C; ++i) {
          size_t e = (size_t)c * C + i;
          float v = owner[e];
          for (int q = 1; q <= K; ++q) v = v + acc[(size_t)mod(c + q, K) * N + e];
          owner[e] = v;
        }
      continue;
    }
    st = oracle_reduce_scatter_sim(ptrs, K, N, ORC_F32, 1.0f, sp, NULL);
    if (st) break;
    if (g_mutation == MUT_PIPE_SCALE_PER_GROUP)
      for (size_t i = 0; i < (size_t)K * C; ++i) sg[i] = apply_scale(sg[i], scale);
    if (g_mutation != MUT_PIPE_REVERSED_GROUPS)
      for (size_t i = 0; i < (size_t)K * C; ++i) owner[i] = owner[i] + sg[i];
  }
  if (!st && g_mutation == MUT_PIPE_REVERSED_GROUPS)
    for (int g = G - 1; g >= 0; --g)
      for (size_t i = 0; i < (size_t)K * C; ++i) owner[i] = owner[i] + settled[(size_t)g * K * C + i];
  for (int c = 0; !st && c < K; ++c)
    for (size_t i = 0; i < C; ++i) {
      float v = owner[(size_t)c * C + i];
      if (g_mutation != MUT_PIPE_SCALE_PER_GROUP) v = apply_scale(v, scale);
      if (out_f32) out_f32[c][i] = v;
      if (out_bf16) out_bf16[c][i] = bf16_round(v);
    }
  free(acc); free(owner); free(settled); free(ptrs); free(sp);
  return st;
}
