/*
 * dp.h -- C ABI of the GB300 (sm_103a) data-parallel collective data path.
 *
 * K data-parallel ranks are "virtual": K rank buffers that live in the one
 * GPU's device memory.  Every call enqueues hand-written CUDA kernels on the
 * caller's stream and returns; no call synchronises, except
 * dp_get_device_error().
 *
 * Shared conventions
 * ------------------
 *  - Pointer arrays (bufs, shards, out_*, w_shards, grads) are HOST arrays
 *    whose entries are DEVICE pointers, one per rank, in the manner of the
 *    per-device send/receive buffers of an NCCL all-reduce ("CMU 11-868
 *    L14-L15: Distributed Training and Data Parallelism, and Where Gradient
 *    Sync Costs Come From", section "NCCL's five building blocks" and the
 *    ncclAllReduce listing after "Ring AllReduce: ReduceScatter, then
 *    AllGather").  The host arrays are read during the call only; the
 *    pointers are passed by value to the kernels, so no host->device copy
 *    happens and the caller may reuse the host array at once.
 *  - Ownership: the caller owns all memory; no call allocates device memory.
 *    The library's state is a 4-byte device error word and the 8 MiB scratch
 *    array of dp_wgrad_reduce_scatter_noalloc (file-scope __device__
 *    variables, placed by the CUDA runtime when it loads the library), a
 *    cached driver entry point, four streams with their events per device
 *    for dp_all_gather_copy_engine (created on its first call), and the
 *    host-side bookkeeping (with their own streams and events) of the
 *    reducer and settle-pipe objects the caller creates and destroys.
 *  - Chunks: a rank buffer of N elements is split into K chunks of
 *    C = ceil(N/K) elements; chunk c is [c*C, min((c+1)*C, N)) (the page's
 *    "each worker splits its gradient into K chunks").
 *  - Ring order: the reduced chunk c ends on rank c and is the fp32 left
 *    fold x_{c+1} + x_{c+2} + ... + x_{c} (rank indices mod K): at step s
 *    rank r passes chunk (r-s-1) mod K to rank r+1, which adds it to its own
 *    matching chunk (section "Ring AllReduce: ReduceScatter, then
 *    AllGather").  Results are bit-identical to that ring for every input,
 *    because the kernels keep this order for every element.
 *  - Arithmetic: bf16 inputs are widened exactly to fp32; the fold is fp32
 *    round-to-nearest-even; `scale` (1/K for the average of "Intuition: data
 *    parallelism has only one thing to synchronize", step 3) multiplies the
 *    folded fp32 value once; the result is rounded once to the output type
 *    (bf16: round-to-nearest-even).
 *  - Limits: 1 <= K <= DP_MAX_K.  N == 0 is a no-op returning DP_OK.
 *  - Memory: any address the GPU can dereference -- device memory, or pinned
 *    host memory (cudaHostAlloc / cudaMallocHost), which the kernels then
 *    read and write across the host link (zero-copy).  The alias checks
 *    compare addresses only.
 *  - Alignment: any element-aligned pointer is accepted; 16-byte-aligned
 *    buffers (with 16-byte-aligned chunk starts) take the vector path,
 *    anything else a slower scalar path with the same results.
 *  - Errors: a status is returned; DP_ERR_CUDA means a launch failed (the
 *    CUDA error is left for cudaGetLastError to report).  Invalid arguments
 *    are rejected before anything is enqueued.
 *  - Threads: every entry point is reentrant and may be called from several
 *    host threads (dp_wgrad_reduce_scatter_noalloc shares one scratch array:
 *    its calls must not overlap on the GPU).
 */
#ifndef DP_GB300_H
#define DP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DP_API __attribute__((visibility("default")))
#else
#define DP_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* dp_stream_t;

typedef enum {
  DP_OK = 0,
  DP_ERR_INVALID_ARG = 1, /* null pointer, K out of range, N % K != 0, ...   */
  DP_ERR_UNSUPPORTED = 2, /* dtype or shape this entry point does not take   */
  DP_ERR_ALIAS = 3,       /* buffers that must be disjoint overlap           */
  DP_ERR_CUDA = 4,        /* a CUDA call failed (no device, launch failure)  */
  DP_ERR_TIMEOUT = 5      /* a bounded device-side wait expired (see below)  */
} dp_status_t;

typedef enum { DP_FP32 = 0, DP_BF16 = 1 } dp_dtype_t;

#define DP_MAX_K 16
#define DP_MAX_MICROBATCHES 16

/*
 * Ring all-reduce, in place ("CMU 11-868 L14-L15 ...", section "Ring
 * AllReduce: ReduceScatter, then AllGather": the reduce-scatter phase, then
 * the all-gather phase; section "NCCL's five building blocks": AllReduce =
 * ReduceScatter + AllGather; ring bound T_AR >= 2B(X-1)/(XW) in "Sharding
 * and Parallelism", section "The cost of the inserted collectives").
 *
 * bufs: K device buffers of N elements of `dtype`, pairwise disjoint.
 * After the call every bufs[r][e] = cast(scale * fold_c(e)), with c the chunk
 * of e.  Any N (C = ceil(N/K); trailing chunks may be short or empty).
 * One kernel reads and writes every element once.
 * Errors: DP_ERR_INVALID_ARG (null, K), DP_ERR_UNSUPPORTED (dtype),
 * DP_ERR_ALIAS (two ranks' buffers overlap), DP_ERR_CUDA.
 */
DP_API dp_status_t dp_ring_allreduce(void* const* bufs, int K, size_t N, dp_dtype_t dtype, float scale,
                              dp_stream_t stream);

/*
 * Ring reduce-scatter ("CMU 11-868 L14-L15 ...", section "Ring AllReduce:
 * ReduceScatter, then AllGather", phase 1; the FSDP backward's per-layer
 * gradient reduce-scatter of "Using ODC to Accelerate AMD SFT Training",
 * section "Why FSDP is Slow"; bound T_RS >= B(X-1)/(XW) in "Sharding and
 * Parallelism", section "The cost of the inserted collectives").
 *
 * bufs: K device buffers of N elements of in_dtype (not modified).
 * out_shards: K device buffers of N/K elements of out_dtype; out_shards[c]
 * receives cast(scale * fold_c) for chunk c (rank c's shard).
 * Requires N % K == 0 (even partition; padding indivisible sizes is the
 * caller's job).  Outputs must not overlap inputs or each other.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_reduce_scatter(const void* const* bufs, int K, size_t N, dp_dtype_t in_dtype,
                              void* const* out_shards, float scale, dp_dtype_t out_dtype,
                              dp_stream_t stream);

/*
 * Ring reduce-scatter emitting both an fp32 and a bf16 shard from the same
 * scaled fp32 value, reading the inputs once (the FSDP gradient
 * reduce-scatter with a master-precision and a compute-precision copy; the
 * page "Sharding and Parallelism", section "Communication predictions",
 * notes that fp32 gradients double the bf16 byte counts).
 *
 * out_f32 (K buffers of N/K floats) or out_bf16 (K buffers of N/K bf16) may
 * be NULL, not both.  Otherwise as dp_reduce_scatter.
 */
DP_API dp_status_t dp_reduce_scatter_dual(const void* const* bufs, int K, size_t N, dp_dtype_t in_dtype,
                                   float* const* out_f32, void* const* out_bf16, float scale,
                                   dp_stream_t stream);

/*
 * Ring all-gather ("CMU 11-868 L14-L15 ...", section "Ring AllReduce:
 * ReduceScatter, then AllGather", phase 2; FSDP's parameter all-gather in
 * "Using ODC to Accelerate AMD SFT Training", section "Why FSDP is Slow";
 * bound T_AG >= B(X-1)/(XW) in "Sharding and Parallelism", section "The
 * cost of the inserted collectives").
 *
 * shards: K device buffers of shard_elems elements of dtype (rank c's
 * finished chunk c).  out: K device buffers of K*shard_elems elements; each
 * receives shard_0 .. shard_{K-1} concatenated, bit for bit.  Outputs must
 * not overlap each other or the shards.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_all_gather(const void* const* shards, int K, size_t shard_elems, dp_dtype_t dtype,
                          void* const* out, dp_stream_t stream);

/*
 * FSDP forward: parameter all-gather fused into the local matmul ("Sharding
 * and Parallelism", section "Real HLO before and after partitioning": the
 * partitioned program all-gathers w[64,512] shards to w[512,512] before the
 * local dot with x[128,512]; section "FSDP and ZeRO": the forward pass
 * gathers W before the dot).
 *
 * x_local: device, row-major [M, D] bf16.  w_shards: K device buffers,
 * each row-major [F_shard, D] bf16; row f of the gathered weight w[F, D]
 * (F = K*F_shard) is row f mod F_shard of shard f / F_shard.  y: device,
 * row-major [M, F] of y_dtype (DP_BF16 or DP_FP32):
 *   y[m, f] = sum_d x[m, d] * w[f, d]   (y = x . w^T),
 * bf16 products accumulated in fp32 on the tensor cores; the gathered w is
 * never materialised (tiles are loaded by TMA straight from the shards).
 * Requires D % 8 == 0 and F_shard % 16 == 0, all base pointers 16-byte
 * aligned, M, D, F_shard < 2^31.  y must not overlap the operands.
 * The summation order over d is the tensor core's, so y matches an fp64
 * reference to within fp32 accumulation error, not bit for bit.
 *
 * workspace (optional, NULL / 0 bytes: none): caller-owned device memory of
 * workspace_bytes, 16-byte aligned, overlapping no operand or output, any
 * contents.  With at least dp_allgather_matmul_workspace_size() bytes, the
 * output tiles of a last round of the persistent grid that is at most half
 * full have their k-blocks split between several otherwise idle CTAs that
 * hand the fp32 accumulator on
 * through the workspace (the same chained split as dp_wgrad_reduce_scatter:
 * the result is bitwise the same with or without it, under any CTA limit).
 * Calls that may overlap on the GPU need separate workspaces.  Flags carry
 * a per-call value as for dp_wgrad_reduce_scatter: no clearing between
 * calls; after a captured call's replay reported DP_ERR_TIMEOUT, zero the
 * workspace before replaying again.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED (shape/alignment, or a
 * device that is not sm_103), DP_ERR_ALIAS, DP_ERR_CUDA; DP_ERR_TIMEOUT is
 * reported later by dp_get_device_error if a pipeline wait expired.
 */
DP_API dp_status_t dp_allgather_matmul(const void* x_local, int M, int D, const void* const* w_shards,
                                int K, int F_shard, void* y, dp_dtype_t y_dtype,
                                void* workspace, size_t workspace_bytes, dp_stream_t stream);

/*
 * Workspace bytes with which dp_allgather_matmul(M, D, K, F_shard) splits its
 * last round on the current device under the current CTA limit; 0 when the
 * shape has no last round at most half full.  A smaller workspace is not an
 * error: the call then runs without the split.
 * Errors: DP_ERR_INVALID_ARG (bytes NULL, K out of range, negative sizes),
 * DP_ERR_CUDA (no device).
 */
DP_API dp_status_t dp_allgather_matmul_workspace_size(int M, int D, int K, int F_shard,
                                                      size_t* bytes);

/*
 * Tensor-parallel partial products summed across the ranks, fused into one
 * GEMM ("Sharding and Parallelism", section "Real HLO before and after
 * partitioning", TP-style fixture: the contracting dimension of both
 * operands is split over the ranks, each computes a partial dot, and an
 * eight-way all-reduce sums the partials; section "Parallelism strategies":
 * tensor parallelism communicates by AllReduce or AllGather/ReduceScatter).
 *
 * Rank r holds x_shards[r]: device, row-major [M, D_shard] bf16, and
 * w_shards[r]: device, row-major [F, D_shard] bf16 (the weight in the
 * [out, in] layout, so both operands are contiguous along the contracted
 * dimension).  The result is
 *   y[m, f] = scale * sum_r sum_d x_r[m, d] * w_r[f, d]
 * with every partial product accumulated in the same fp32 tensor-core
 * accumulator (the psum happens in TMEM; the partials are never written).
 *
 * dp_matmul_allreduce: y_out holds K device buffers [M, F] of y_dtype; every
 *   rank's buffer receives the whole result.
 * dp_matmul_reduce_scatter: requires M % K == 0; y_out[c] is a device buffer
 *   [M/K, F] receiving rows [c*M/K, (c+1)*M/K) -- chunk c of the row-major
 *   result, as the ring reduce-scatter of the flattened partials would leave
 *   on rank c.
 * Requires D_shard % 8 == 0, F % 16 == 0, 16-byte-aligned base pointers;
 * outputs must not overlap the operands or each other.  Accuracy as for
 * dp_allgather_matmul (fp32 accumulation, not bit-defined).  workspace /
 * workspace_bytes: optional, as for dp_allgather_matmul (size from
 * dp_matmul_workspace_size; bitwise the same result with or without).
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_matmul_allreduce(const void* const* x_shards, const void* const* w_shards,
                                       int K, int M, int D_shard, int F, void* const* y_out,
                                       dp_dtype_t y_dtype, float scale, void* workspace,
                                       size_t workspace_bytes, dp_stream_t stream);
DP_API dp_status_t dp_matmul_reduce_scatter(const void* const* x_shards,
                                            const void* const* w_shards, int K, int M,
                                            int D_shard, int F, void* const* y_out,
                                            dp_dtype_t y_dtype, float scale, void* workspace,
                                            size_t workspace_bytes, dp_stream_t stream);

/*
 * The same two calls in the x . w orientation of the page's fixture ("Sharding
 * and Parallelism", section "Real HLO before and after partitioning", TP-style
 * fixture x[1024,64] @ w[64,512] per rank: the weight is sharded along its
 * contracted rows): w_shards[r] is device, row-major [D_shard, F] bf16, and
 *   y[m, f] = scale * sum_r sum_d x_r[m, d] * w_r[d, f].
 * The tensor core reads w_r column-major from shared memory (the
 * instruction's B transpose), so nothing is transposed in memory.  Requires
 * F % 64 == 0 in addition to the conditions of dp_matmul_allreduce; outputs,
 * workspace (size from dp_matmul_xw_workspace_size) and errors as there.
 */
DP_API dp_status_t dp_matmul_allreduce_xw(const void* const* x_shards,
                                          const void* const* w_shards, int K, int M,
                                          int D_shard, int F, void* const* y_out,
                                          dp_dtype_t y_dtype, float scale, void* workspace,
                                          size_t workspace_bytes, dp_stream_t stream);
DP_API dp_status_t dp_matmul_reduce_scatter_xw(const void* const* x_shards,
                                               const void* const* w_shards, int K, int M,
                                               int D_shard, int F, void* const* y_out,
                                               dp_dtype_t y_dtype, float scale, void* workspace,
                                               size_t workspace_bytes, dp_stream_t stream);
DP_API dp_status_t dp_matmul_xw_workspace_size(int K, int M, int D_shard, int F, size_t* bytes);

/*
 * Workspace bytes with which dp_matmul_allreduce / dp_matmul_reduce_scatter
 * (K, M, D_shard, F) split their last round on the current device under the
 * current CTA limit (the two forms share their tiling); 0 when there is no
 * last round at most half full.  Errors as dp_allgather_matmul_workspace_size.
 */
DP_API dp_status_t dp_matmul_workspace_size(int K, int M, int D_shard, int F, size_t* bytes);

/*
 * The FSDP backward weight gradient fused with its reduce-scatter ("Using
 * ODC to Accelerate AMD SFT Training", section "Why FSDP is Slow": in the
 * backward pass each layer computes its full gradient and reduce-scatters it
 * to the rank's shard; "Sharding and Parallelism", section "Real HLO before
 * and after partitioning": an FSDP training step's backward adds a gradient
 * ReduceScatter).  For a linear layer y = x . w^T with w [F, D], rank r's
 * local weight gradient is dW_r = dY_r^T . X_r over its own T tokens, and the
 * data-parallel gradient is their sum ("CMU 11-868 L14-L15", section
 * "Intuition: data parallelism has only one thing to synchronize").
 *
 * Rank r holds dy[r]: device, row-major [T, F] bf16 (the layer's output
 * gradients, tokens x output features) and x[r]: device, row-major [T, D]
 * bf16 (its inputs).  The result is
 *   dW[f, d] = scale * sum_r sum_t dy_r[t, f] * x_r[t, d]
 * with every rank's products accumulated in the same fp32 tensor-core
 * accumulator (the per-rank dW_r are never written).  dw_shards[c] is a
 * device buffer [F/K, D] of dw_dtype receiving rows [c*F/K, (c+1)*F/K) of
 * dW -- chunk c of the row-major gradient, as the ring reduce-scatter of the
 * flattened dW_r would leave on rank c.  scale = 1/K averages.
 * Requires F % K == 0, F % 64 == 0, D % 64 == 0, 16-byte-aligned base
 * pointers; outputs must not overlap the operands or each other.  T == 0
 * writes zeros.  Accuracy as for dp_allgather_matmul (fp32 accumulation, not
 * bit-defined).
 *
 * workspace (optional, NULL / 0 bytes: none): caller-owned device memory of
 * workspace_bytes, 16-byte aligned, not overlapping the operands or outputs,
 * any contents.  With at least dp_wgrad_workspace_size() bytes, the output
 * tiles of a last, less-than-half-full round of the persistent grid have
 * their token blocks split between several CTAs, which hand the fp32
 * accumulator on through the workspace, so that round takes a fraction of a
 * tile's time.  The accumulation order is unchanged: the result is bitwise
 * the same with or without a workspace (and under any CTA limit).  Calls
 * that may overlap on the GPU need separate workspaces.  Each call tags its
 * hand-off flags with a 64-bit value of its own and clears each flag once
 * it is read, so the workspace needs no clearing between calls.  A replay
 * of a captured call reuses the captured value: after a replay whose wait
 * expired (DP_ERR_TIMEOUT), zero the workspace before replaying again.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA;
 * DP_ERR_TIMEOUT (from dp_get_device_error) if a hand-off waited > 2 s.
 */
DP_API dp_status_t dp_wgrad_reduce_scatter(const void* const* dy, const void* const* x, int K,
                                           int T, int F, int D, void* const* dw_shards,
                                           dp_dtype_t dw_dtype, float scale, void* workspace,
                                           size_t workspace_bytes, dp_stream_t stream);

/*
 * Workspace bytes with which dp_wgrad_reduce_scatter(K, T, F, D) splits its
 * last round on the current device under the current CTA limit
 * (dp_set_cta_limits); 0 when the shape has no such round.  A smaller
 * workspace is not an error: the call then runs without the split.
 * Errors: DP_ERR_INVALID_ARG (bytes NULL, K out of range, negative sizes),
 * DP_ERR_CUDA (no device).
 */
DP_API dp_status_t dp_wgrad_workspace_size(int K, int T, int F, int D, size_t* bytes);

/*
 * The paper has no counterpart to this call: it exists for callers that
 * cannot allocate device memory.  Frameworks whose memory pool owns the GPU
 * may forbid allocations outside the pool; a training step may not afford
 * the device-wide synchronisation that cudaMalloc / cudaFree can cause; a
 * deployment may fix its device-memory budget at start-up.  Such callers
 * cannot hand dp_wgrad_reduce_scatter a workspace, and would lose its split
 * of a part-full last round.
 *
 * dp_wgrad_reduce_scatter_noalloc computes exactly what dp_wgrad_reduce_scatter
 * does with a sufficient workspace (same arguments, same result bits), taking
 * the scratch from a file-scope device array of DP_WGRAD_NOALLOC_MAX_BYTES
 * (8 MiB) that every GPU which loads this library holds until the process
 * exits.  The call allocates nothing.  It rejects a shape whose split would
 * need more scratch than that (dp_wgrad_workspace_size() > the maximum) with
 * DP_ERR_UNSUPPORTED, without launching; shapes that need no scratch run
 * unsplit.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Every call on a device shares the one array,
 * which keeps the previous call's contents; none of it needs clearing,
 * because each call tags its hand-off flags with a 64-bit value of its own
 * and reads a partial sum only after its flag carries that value.  Calls
 * that may overlap on the GPU race on the array and give wrong results.
 * Otherwise as dp_wgrad_reduce_scatter.
 * Errors: as dp_wgrad_reduce_scatter, plus DP_ERR_UNSUPPORTED when the
 * scratch needed exceeds DP_WGRAD_NOALLOC_MAX_BYTES.
 */
#define DP_WGRAD_NOALLOC_MAX_BYTES ((size_t)8 << 20)
DP_API dp_status_t dp_wgrad_reduce_scatter_noalloc(const void* const* dy, const void* const* x,
                                                   int K, int T, int F, int D,
                                                   void* const* dw_shards, dp_dtype_t dw_dtype,
                                                   float scale, dp_stream_t stream);

/*
 * One microbatch into a rank's fp32 gradient accumulator ("Using ODC to
 * Accelerate AMD SFT Training", section "From Per-iteration to Per-minibatch
 * Synchronization": microbatch gradients are accumulated locally and settled
 * once per minibatch; section "odc_pad vs odc_nopad", Figure 5: padding
 * buckets contribute no valid gradient).
 *
 * acc: device, N floats.  grad: device, N elements of grad_dtype, or NULL
 * for a padding bucket (gradient +0; the accumulator is still read and
 * rewritten, as a padded microbatch still costs its pass).
 *   acc[e] = (first ? +0 : acc[e]) + widen(grad[e]).
 * The accumulator starts at +0, so a padding bucket never changes its bits.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_grad_accumulate(float* acc, const void* grad, size_t N, dp_dtype_t grad_dtype,
                               int first, dp_stream_t stream);

/*
 * The variable-length step's accumulate and settle in one pass ("Using ODC
 * to Accelerate AMD SFT Training", sections "From Per-iteration to
 * Per-minibatch Synchronization" and "odc_pad vs odc_nopad").
 *
 * grads: HOST table of K*Mmax device pointers, row-major by rank
 * (grads[r*Mmax + j] is microbatch j of rank r, N elements of grad_dtype,
 * or NULL for a padding bucket).  m: HOST array of K counts, 0 <= m[r] <=
 * Mmax <= DP_MAX_MICROBATCHES.  Rank r's gradient is the fp32 sum
 * (+0) + g_{r,0} + ... + g_{r,m[r]-1}, in that order; the K sums are then
 * ring-reduce-scattered exactly as dp_reduce_scatter_dual with in_dtype
 * DP_FP32 would do on K accumulators built by dp_grad_accumulate, without
 * writing the accumulators.  Requires N % K == 0.  out_f32 / out_bf16 as in
 * dp_reduce_scatter_dual.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_odc_reduce_scatter(const void* const* grads, const int* m, int K, int Mmax,
                                  size_t N, dp_dtype_t grad_dtype, float* const* out_f32,
                                  void* const* out_bf16, float scale, dp_stream_t stream);

/*
 * All-reduce of one DDP gradient bucket, in place, without flattening it
 * ("CMU 11-868 L14-L15 ...", section "When to sync: gradient bucketing":
 * gradients are grouped into buckets and each bucket is all-reduced as one
 * message).
 *
 * The bucket is the concatenation, in the given order, of n tensors; tensor t
 * has numels[t] elements of dtype and its K rank copies are
 * grads[t*K + r] (HOST array of n*K device pointers).  The result equals a
 * ring all-reduce of the flat bucket of total = sum numels elements: chunk
 * length C = ceil(total/K), an element at bucket offset o is folded in the
 * order of chunk o / C, scaled, cast and written back into every rank's copy.
 * All n*K buffers must be pairwise disjoint.  Any alignment and any sizes
 * (16-byte-aligned tensors take the vector path); a tensor with numels[t] ==
 * 0 takes no part, and its pointers may be NULL (as frameworks give empty
 * tensors), every other pointer must not be.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_bucket_allreduce(void* const* grads, const size_t* numels, int n, int K,
                                       dp_dtype_t dtype, float scale, dp_stream_t stream);

/*
 * One microbatch group's settle in a cross-iteration settle pipeline ("Using
 * ODC to Accelerate AMD SFT Training", section "Discussion: Settle Does Not
 * Yet Overlap with Backward": the previous microbatch group's settle runs on
 * a separate stream beside this group's backward compute, joined once per
 * minibatch; the settle itself as in "From Per-iteration to Per-minibatch
 * Synchronization").
 *
 * A minibatch's microbatches are split into groups, index ranges of j shared
 * by the ranks.  grads / m / Mmax describe this group only, as for
 * dp_odc_reduce_scatter: m[r] (0 allowed) of rank r's microbatches, in
 * order.  Each rank's group sum (+0) + g_{r,j} + ... is ring-folded over the
 * ranks exactly as dp_odc_reduce_scatter does, giving the settled chunk S_c
 * (not yet averaged).  owner_acc: HOST array of K device pointers, chunk c's
 * fp32 running sum (N/K floats each, caller-owned, 16-byte aligned for the
 * vector path).  phase (bits):
 *   DP_SETTLE_FIRST            owner_acc[c] = +0 + S_c    (outputs unused)
 *   0                          owner_acc[c] = owner_acc[c] + S_c
 *   DP_SETTLE_LAST             out[c] = cast((owner_acc[c] + S_c) * scale)
 *   DP_SETTLE_FIRST|LAST       out[c] = cast(S_c * scale) (= dp_odc_reduce_scatter;
 *                              owner_acc may be NULL)
 * so the owner adds the groups' settled chunks in the order of the calls and
 * averages once.  out_f32 / out_bf16 as in dp_reduce_scatter_dual (required
 * only with DP_SETTLE_LAST).  owner_acc must not overlap the gradients or
 * the outputs.  Requires N % K == 0.
 * Errors: DP_ERR_INVALID_ARG (also: phase outside the two bits, owner_acc
 * NULL when a phase needs it), DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
#define DP_SETTLE_FIRST 1
#define DP_SETTLE_LAST 2
DP_API dp_status_t dp_odc_settle_group(const void* const* grads, const int* m, int K, int Mmax,
                                       size_t N, dp_dtype_t grad_dtype, float* const* owner_acc,
                                       int phase, float* const* out_f32, void* const* out_bf16,
                                       float scale, dp_stream_t stream);

/*
 * The cross-iteration settle pipeline: a side stream and events that run
 * each pushed group settle beside the caller's compute, and one join per
 * minibatch ("Using ODC to Accelerate AMD SFT Training", section
 * "Discussion: Settle Does Not Yet Overlap with Backward").
 *
 * dp_settle_pipe_create: a pipe on the current device, with its own
 *   non-blocking stream and two events (the library's only allocations here:
 *   CUDA stream and event objects, no device memory).  cta_limit > 0 caps
 *   the CTAs of the pipe's settle launches (so the compute keeps the other
 *   SMs), on top of the process-wide limit of dp_set_cta_limits; 0: that
 *   limit alone.
 * dp_settle_pipe_push: the group's gradients are complete in `stream`'s
 *   order at this point; the call records that point, makes the pipe's
 *   stream wait for it and enqueues dp_odc_settle_group (same arguments) on
 *   the pipe's stream, then returns; work enqueued afterwards on `stream`
 *   (the next group's backward) runs concurrently with the settle.  Settles
 *   run in push order.  The pushed gradient buffers are read until the
 *   settle finishes: do not overwrite them before a dp_settle_pipe_wait.
 *   Arguments are validated before anything is enqueued.
 * dp_settle_pipe_wait: `stream` waits for every settle pushed so far (the
 *   once-per-minibatch join; afterwards the outputs, the owners'
 *   accumulators and the pushed gradient buffers are free to use in
 *   `stream`'s order).  Under stream capture, join before ending the
 *   capture.
 * dp_settle_pipe_destroy: waits for the pipe's stream, then frees it.
 * Pushes and waits from several threads are serialised per pipe; the
 * current device must be the pipe's.
 * Errors: DP_ERR_INVALID_ARG (NULL pipe, another device), the errors of
 * dp_odc_settle_group, DP_ERR_CUDA.
 */
typedef struct dp_settle_pipe dp_settle_pipe_t;
DP_API dp_status_t dp_settle_pipe_create(int cta_limit, dp_settle_pipe_t** pipe);
DP_API dp_status_t dp_settle_pipe_push(dp_settle_pipe_t* pipe, const void* const* grads,
                                       const int* m, int K, int Mmax, size_t N,
                                       dp_dtype_t grad_dtype, float* const* owner_acc, int phase,
                                       float* const* out_f32, void* const* out_bf16, float scale,
                                       dp_stream_t stream);
DP_API dp_status_t dp_settle_pipe_wait(dp_settle_pipe_t* pipe, dp_stream_t stream);
DP_API dp_status_t dp_settle_pipe_destroy(dp_settle_pipe_t* pipe);

/*
 * The DDP gradient Reducer (same sections of "CMU 11-868 L14-L15 ...":
 * bucket_cap_mb, the fixed parameter-to-bucket map, reverse parameter order,
 * pending counts, buckets launched strictly in order, unused parameters).
 *
 * dp_reducer_create: P parameters of numels[p] elements of dtype, K ranks,
 *   bucket cap in bytes (25 MB = 25*1024*1024 in DDP's default), scale for
 *   every bucket's all-reduce (1/K averages).  Parameters are walked from
 *   P-1 down to 0 and appended to the open bucket, which is closed as soon as
 *   its size reaches the cap.  *out receives an opaque host object.
 * dp_reducer_mark_ready: parameter p's gradient is ready on all K ranks at
 *   grads[0..K-1] (HOST array of device pointers, read during the call;
 *   NULL is accepted only for a parameter of 0 elements).
 *   Decrements p's bucket's pending count; then every consecutive complete
 *   bucket from the next unlaunched one onward is all-reduced on `stream`
 *   (dp_bucket_allreduce over its parameters, in bucket layout order), and
 *   *launched (nullable) receives how many were launched by this call.
 *   Marking a parameter twice in one iteration is DP_ERR_INVALID_ARG.
 * dp_reducer_finish: ends the iteration.  DP_OK if every bucket was launched;
 *   otherwise DP_ERR_INVALID_ARG with *first_pending = the first bucket that
 *   never completed (a parameter that took no part -- where DDP would hang).
 *   Either way the reducer is reset for the next iteration.
 * dp_reducer_bucket_info / dp_reducer_param_slot: the layout (bucket sizes,
 *   parameter -> (bucket, element offset in the bucket)).
 * dp_reducer_set_dry_run: when on, buckets are recorded but not launched
 *   (lets the host logic be exercised without a GPU);
 *   dp_reducer_launch_log copies this iteration's launched bucket ids.
 * dp_reducer_set_overlap: on != 0 makes the reducer create (on the current
 *   device) two non-blocking streams of its own and three events; from then
 *   on bucket b is all-reduced on stream b % 2, after an event recorded in
 *   the mark_ready call's `stream` at the point where the bucket completed,
 *   so the caller's stream goes on with the backward of earlier layers while
 *   the bucket is reduced ("When to sync: gradient bucketing": the Reducer
 *   launches an asynchronous AllReduce while backward keeps computing), and
 *   consecutive buckets, whose data are disjoint, may run at the same time.
 *   on == 0 waits for and frees them.  mark_ready must then be called with
 *   that device current.
 * dp_reducer_wait: `stream` waits for every bucket launched so far (the
 *   join before the optimizer step reads the gradients); DP_OK and nothing
 *   to do without overlap.  In overlap mode the gradients of a launched
 *   bucket must not be written again before this join.
 * dp_reducer_destroy also waits for the reducer's streams.
 * A reducer is used by one iteration at a time; its calls are serialised by
 * an internal mutex.
 */
typedef struct dp_reducer dp_reducer_t;
DP_API dp_status_t dp_reducer_create(const size_t* numels, int P, dp_dtype_t dtype, int K,
                                     size_t bucket_cap_bytes, float scale, dp_reducer_t** out);
DP_API void dp_reducer_destroy(dp_reducer_t* r);
DP_API int dp_reducer_num_buckets(const dp_reducer_t* r);
DP_API dp_status_t dp_reducer_bucket_info(const dp_reducer_t* r, int b, int* num_params,
                                          size_t* numel);
DP_API dp_status_t dp_reducer_param_slot(const dp_reducer_t* r, int p, int* bucket,
                                         size_t* offset);
DP_API dp_status_t dp_reducer_mark_ready(dp_reducer_t* r, int p, void* const* grads,
                                         dp_stream_t stream, int* launched);
DP_API dp_status_t dp_reducer_finish(dp_reducer_t* r, int* first_pending);
DP_API dp_status_t dp_reducer_set_dry_run(dp_reducer_t* r, int on);
DP_API int dp_reducer_launch_log(dp_reducer_t* r, int* buckets, int cap);
DP_API dp_status_t dp_reducer_set_overlap(dp_reducer_t* r, int on);
DP_API dp_status_t dp_reducer_wait(dp_reducer_t* r, dp_stream_t stream);

/*
 * The parameter all-gather on the GPU's copy engines instead of its SMs
 * ("Optimizing ML Concurrent Computation and Communication with GPU DMA
 * Engines", Q2 "ConCCL (DMA Offload)": collectives that only move data can
 * run on DMA engines so that a concurrent GEMM keeps every compute unit).
 * Same arguments and result as dp_all_gather: K*K device-to-device
 * cudaMemcpyAsync copies (destination rank r, shard c), no kernel.  The
 * copies run on four internal streams of the library (created, with their
 * events, on the first call on each device: make that call before any stream
 * capture), forked from `stream` and joined back to it through events, so
 * several DMA engines work at once (issued shard by shard, each engine on
 * another destination of the same shard, so that repeated reads of a shard
 * hit L2) and the result is ordered on `stream` like any other call.  Calls
 * from several host
 * threads are serialised while they issue.  Bit-identical to dp_all_gather.
 * Errors: DP_ERR_INVALID_ARG, DP_ERR_UNSUPPORTED, DP_ERR_ALIAS, DP_ERR_CUDA.
 */
DP_API dp_status_t dp_all_gather_copy_engine(const void* const* shards, int K,
                                             size_t shard_elems, dp_dtype_t dtype,
                                             void* const* out, dp_stream_t stream);

/*
 * Which implementation dp_ring_allreduce and dp_all_gather use for aligned
 * buffers (process-wide, default 0):
 *   0  automatic: the bulk-copy kernels (the faster on GB300), except an
 *      all-reduce of at most 32 KiB per rank, which starts sooner on the
 *      register kernel;
 *   1  registers: every thread loads 16-byte vectors from the K ranks, folds
 *      them and stores the result to the K ranks;
 *   2  bulk copies: tiles cross shared memory by cp.async.bulk (TMA) -- K
 *      bulk loads, the fold in shared memory, K bulk stores issued by one
 *      thread per tile (the all-reduce "streamed through shared memory or
 *      TMA once" rather than in K-1 passes); the all-gather gives each CTA
 *      one destination rank (one load, one store per tile; the K ranks'
 *      CTAs read each tile together, so DRAM serves it once), or, under a
 *      stream CTA limit, one source shard (one load, K stores per tile).
 * The variants give identical bits.  Returns DP_ERR_INVALID_ARG for other
 * values.
 */
DP_API dp_status_t dp_set_collective_variant(int variant);
DP_API int dp_get_collective_variant(void);

/*
 * Process-wide upper bounds on the CTAs one launch may use: gemm_ctas for
 * the tensor-core kernels (dp_allgather_matmul, dp_matmul_*,
 * dp_wgrad_reduce_scatter*; the weight gradient's workspace size follows the
 * limit), stream_ctas
 * for the streaming collectives (reduce-scatter, all-gather, all-reduce,
 * accumulate, bucket and variable-length kernels); 0 means no limit (the
 * default: one resident grid over every SM).  Lets a caller leave SMs free
 * for a kernel on another stream -- the resource-partitioning experiment of
 * "Optimizing ML Concurrent Computation and Communication with GPU DMA
 * Engines" (Q2, "Resource Partitioning").  Results do not depend on the
 * limits.  Applies to launches made after the call, from any thread.
 */
DP_API dp_status_t dp_set_cta_limits(int gemm_ctas, int stream_ctas);
DP_API dp_status_t dp_get_cta_limits(int* gemm_ctas, int* stream_ctas);

/*
 * Synchronises `stream`, then reports and clears the device error word of
 * the current device: DP_ERR_TIMEOUT if a bounded device-side wait expired
 * in any kernel since the last call, DP_ERR_CUDA if the stream reported a
 * CUDA error, DP_OK otherwise.
 */
DP_API dp_status_t dp_get_device_error(dp_stream_t stream);

/*
 * Diagnostic: launches one block that waits, with the library's bounded
 * wait, on a barrier that nothing completes, for at most timeout_us
 * microseconds, then records the expiry in the device error word and
 * returns.  dp_get_device_error then reports DP_ERR_TIMEOUT.  Lets a test
 * exercise the timeout path without touching any other kernel.
 * timeout_us must be in [1, 2000000].
 */
DP_API dp_status_t dp_selftest_bounded_wait(uint32_t timeout_us, dp_stream_t stream);

/* Static, human-readable name of a status. */
DP_API const char* dp_status_string(dp_status_t s);

/* Library version as 10000*major + 100*minor + patch. */
DP_API int dp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DP_GB300_H */
