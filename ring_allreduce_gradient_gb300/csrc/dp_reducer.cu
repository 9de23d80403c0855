// dp_reducer.cu -- the DDP gradient Reducer (host side) and the bucket
// all-reduce entry point.
//
// "CMU 11-868 L14-L15: Distributed Training and Data Parallelism, and Where
// Gradient Sync Costs Come From", sections "When to sync: gradient bucketing"
// and "What the paper adds beyond the slides":
//  * the parameter -> bucket mapping is fixed at construction from the size
//    limit (bucket_cap_mb, 25 MB by default) and the parameter sizes;
//  * parameters enter buckets in the reverse order of model.parameters(),
//    since backward produces gradients roughly in that order;
//  * each gradient's readiness decrements its bucket's pending count; a
//    bucket whose count reaches zero is all-reduced, and buckets are launched
//    strictly in bucket order (bucket i+1 never before bucket i);
//  * a parameter that takes no part in an iteration leaves its bucket
//    incomplete and would hang DDP's backward; here the end-of-iteration
//    check reports the first incomplete bucket instead;
//  * "once every gradient in a bucket is ready, the Reducer launches an
//    asynchronous AllReduce on it while backward keeps computing earlier
//    layers": in overlap mode each bucket is reduced on one of the reducer's
//    own streams, after an event recorded where the bucket completed in the
//    caller's stream, and dp_reducer_wait joins them before the optimizer.
//    Consecutive buckets alternate between two such streams: their data are
//    disjoint, so a bucket's grid can fill the SMs that the previous one's
//    last CTAs leave idle (GPT-2-small gradients, one iteration from a CUDA
//    graph on GB300: 1 MiB buckets 1.374 -> 1.293 ms, 25 MiB 1.244 -> 1.224
//    ms; three or four streams gained no more).
//
// Reading of the size rule: walk the parameters from last to first, append
// each to the open bucket, and close the bucket as soon as its size reaches
// the cap (so one bucket may exceed the cap by its last parameter, and a
// parameter larger than the cap gets a bucket of its own).

#include "dp_launch.h"

#include <algorithm>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

struct dp_reducer {
  int P = 0, K = 0;
  dp_dtype_t dtype = DP_FP32;
  float scale = 1.0f;
  size_t cap_bytes = 0;
  std::vector<size_t> numel;              // per parameter
  std::vector<int> bucket_of;             // per parameter
  std::vector<size_t> offset_in;          // per parameter: element offset inside its bucket
  std::vector<std::vector<int>> members;  // per bucket: parameters in layout order
  std::vector<size_t> bucket_numel;
  // per-iteration state
  std::vector<int> pending;
  std::vector<char> ready;
  std::vector<void*> grads;  // P*K
  int next_bucket = 0;
  bool dry_run = false;
  std::vector<int> launch_log;
  // overlap mode: bucket b is all-reduced on the reducer's stream comm[b % 2],
  // after the point in the caller's stream where it completed
  static constexpr int kComm = 2;
  bool overlap = false;
  int device = -1;
  cudaStream_t comm[kComm] = {};
  cudaEvent_t ev_ready = nullptr;         // a bucket's gradients are complete (caller's stream)
  cudaEvent_t ev_done[kComm] = {};        // every bucket launched so far on comm[i]
  std::mutex mu;
};

namespace {

size_t esize(dp_dtype_t t) { return t == DP_FP32 ? 4u : 2u; }

void reset_iteration(dp_reducer* r) {
  r->pending.assign(r->members.size(), 0);
  for (size_t b = 0; b < r->members.size(); ++b) r->pending[b] = (int)r->members[b].size();
  r->ready.assign(r->P, 0);
  r->next_bucket = 0;
  r->launch_log.clear();
}

dp_status_t launch_bucket(dp_reducer* r, int b, dp_stream_t s) {
  r->launch_log.push_back(b);
  if (r->dry_run) return DP_OK;
  const std::vector<int>& mem = r->members[b];
  std::vector<void*> ptrs(mem.size() * (size_t)r->K);
  std::vector<size_t> ne(mem.size());
  for (size_t i = 0; i < mem.size(); ++i) {
    ne[i] = r->numel[mem[i]];
    for (int k = 0; k < r->K; ++k) ptrs[i * r->K + k] = r->grads[(size_t)mem[i] * r->K + k];
  }
  if (r->overlap) {
    // DDP's asynchronous all-reduce: the caller's stream goes on with the
    // backward of earlier layers while the bucket is reduced on a comm stream
    cudaStream_t c = r->comm[b % dp_reducer::kComm];
    if (cudaEventRecord(r->ev_ready, reinterpret_cast<cudaStream_t>(s)) != cudaSuccess ||
        cudaStreamWaitEvent(c, r->ev_ready, 0) != cudaSuccess) {
      cudaGetLastError();
      return DP_ERR_CUDA;
    }
    s = reinterpret_cast<dp_stream_t>(c);
  }
  return dp_bucket_allreduce(ptrs.data(), ne.data(), (int)mem.size(), r->K, r->dtype, r->scale,
                             s);
}

void release_overlap(dp_reducer* r) {
  for (int i = 0; i < dp_reducer::kComm; ++i)
    if (r->comm[i]) cudaStreamSynchronize(r->comm[i]);
  for (int i = 0; i < dp_reducer::kComm; ++i) {
    if (r->ev_done[i]) cudaEventDestroy(r->ev_done[i]);
    if (r->comm[i]) cudaStreamDestroy(r->comm[i]);
    r->comm[i] = nullptr;
    r->ev_done[i] = nullptr;
  }
  if (r->ev_ready) cudaEventDestroy(r->ev_ready);
  r->ev_ready = nullptr;
  r->overlap = false;
  cudaGetLastError();
}

}  // namespace

extern "C" {

dp_status_t dp_bucket_allreduce(void* const* grads, const size_t* numels, int n, int K,
                                dp_dtype_t dtype, float scale, dp_stream_t stream) {
  dph::NvtxRange nvtx_range("dp_bucket_allreduce");
  if (!grads || !numels || n < 0 || K < 1 || K > DP_MAX_K) return DP_ERR_INVALID_ARG;
  if (dtype != DP_FP32 && dtype != DP_BF16) return DP_ERR_UNSUPPORTED;
  // every rank buffer of every tensor must be present and disjoint from all others
  std::vector<std::pair<uintptr_t, uintptr_t>> rg;
  rg.reserve((size_t)n * K);
  for (int t = 0; t < n; ++t) {
    for (int k = 0; k < K; ++k) {
      void* p = grads[(size_t)t * K + k];
      if (!p && numels[t]) return DP_ERR_INVALID_ARG;  // an empty tensor may be NULL
      const uintptr_t a = reinterpret_cast<uintptr_t>(p);
      if (numels[t]) rg.emplace_back(a, a + numels[t] * esize(dtype));
    }
  }
  std::sort(rg.begin(), rg.end());
  for (size_t i = 1; i < rg.size(); ++i)
    if (rg[i].first < rg[i - 1].second) return DP_ERR_ALIAS;
  if (rg.empty()) return DP_OK;
  dph::DeviceInfo dev;
  if (!dph::current_device(&dev)) return DP_ERR_CUDA;
  dpl::BucketArgs a{grads, numels, n, K, scale, dtype};
  // the bulk-copy kernel needs every tensor 16-byte aligned (any length)
  bool aligned = true;
  for (size_t i = 0; i < (size_t)n * K; ++i)
    aligned = aligned && ((reinterpret_cast<uintptr_t>(grads[i]) & 15u) == 0);
  const int v = dph::collective_variant();
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const bool bulk = aligned && (v == dph::kVariantAuto || v == dph::kVariantBulkCopy);
  const cudaError_t e = bulk ? dpl::launch_bucket_allreduce_tma(a, dev, cs)
                             : dpl::launch_bucket_allreduce(a, dev, cs);
  return e == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}

dp_status_t dp_reducer_create(const size_t* numels, int P, dp_dtype_t dtype, int K,
                              size_t bucket_cap_bytes, float scale, dp_reducer_t** out) {
  if (!out) return DP_ERR_INVALID_ARG;
  *out = nullptr;
  if (!numels || P < 1 || K < 1 || K > DP_MAX_K || bucket_cap_bytes == 0)
    return DP_ERR_INVALID_ARG;
  if (dtype != DP_FP32 && dtype != DP_BF16) return DP_ERR_UNSUPPORTED;
  dp_reducer* r = new (std::nothrow) dp_reducer();
  if (!r) return DP_ERR_INVALID_ARG;
  r->P = P;
  r->K = K;
  r->dtype = dtype;
  r->scale = scale;
  r->cap_bytes = bucket_cap_bytes;
  r->numel.assign(numels, numels + P);
  r->bucket_of.assign(P, -1);
  r->offset_in.assign(P, 0);
  r->grads.assign((size_t)P * K, nullptr);
  std::vector<int> cur;
  size_t cur_elems = 0;
  auto close = [&]() {
    if (cur.empty()) return;
    const int b = (int)r->members.size();
    size_t off = 0;
    for (int p : cur) {
      r->bucket_of[p] = b;
      r->offset_in[p] = off;
      off += r->numel[p];
    }
    r->members.push_back(cur);
    r->bucket_numel.push_back(off);
    cur.clear();
    cur_elems = 0;
  };
  for (int p = P - 1; p >= 0; --p) {
    cur.push_back(p);
    cur_elems += r->numel[p];
    if (cur_elems * esize(dtype) >= bucket_cap_bytes) close();
  }
  close();
  reset_iteration(r);
  *out = r;
  return DP_OK;
}

void dp_reducer_destroy(dp_reducer_t* r) {
  if (!r) return;
  if (r->comm[0]) {
    int prev = -1;
    if (cudaGetDevice(&prev) == cudaSuccess && prev != r->device) cudaSetDevice(r->device);
    release_overlap(r);
    if (prev >= 0 && prev != r->device) cudaSetDevice(prev);
  }
  delete r;
}

dp_status_t dp_reducer_set_overlap(dp_reducer_t* r, int on) {
  if (!r) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(r->mu);
  if (!on) {
    if (r->comm[0]) release_overlap(r);
    return DP_OK;
  }
  if (r->comm[0]) return DP_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DP_ERR_CUDA;
  }
  r->device = dev;
  bool ok = cudaEventCreateWithFlags(&r->ev_ready, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < dp_reducer::kComm; ++i)
    ok = cudaStreamCreateWithFlags(&r->comm[i], cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&r->ev_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release_overlap(r);
    return DP_ERR_CUDA;
  }
  r->overlap = true;
  return DP_OK;
}

dp_status_t dp_reducer_wait(dp_reducer_t* r, dp_stream_t stream) {
  if (!r) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(r->mu);
  if (!r->overlap) return DP_OK;  // buckets ran on the caller's streams
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != r->device) {
    cudaGetLastError();
    return DP_ERR_INVALID_ARG;
  }
  for (int i = 0; i < dp_reducer::kComm; ++i)
    if (cudaEventRecord(r->ev_done[i], r->comm[i]) != cudaSuccess ||
        cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), r->ev_done[i], 0) !=
            cudaSuccess) {
      cudaGetLastError();
      return DP_ERR_CUDA;
    }
  return DP_OK;
}

int dp_reducer_num_buckets(const dp_reducer_t* r) { return r ? (int)r->members.size() : 0; }

dp_status_t dp_reducer_bucket_info(const dp_reducer_t* r, int b, int* num_params,
                                   size_t* numel) {
  if (!r || b < 0 || b >= (int)r->members.size()) return DP_ERR_INVALID_ARG;
  if (num_params) *num_params = (int)r->members[b].size();
  if (numel) *numel = r->bucket_numel[b];
  return DP_OK;
}

dp_status_t dp_reducer_param_slot(const dp_reducer_t* r, int p, int* bucket, size_t* offset) {
  if (!r || p < 0 || p >= r->P) return DP_ERR_INVALID_ARG;
  if (bucket) *bucket = r->bucket_of[p];
  if (offset) *offset = r->offset_in[p];
  return DP_OK;
}

dp_status_t dp_reducer_mark_ready(dp_reducer_t* r, int p, void* const* grads, dp_stream_t stream,
                                  int* launched) {
  dph::NvtxRange nvtx_range("dp_reducer_mark_ready");
  if (launched) *launched = 0;
  if (!r || !grads || p < 0 || p >= r->P) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(r->mu);
  if (r->ready[p]) return DP_ERR_INVALID_ARG;  // marked twice in one iteration
  if (r->overlap && !r->dry_run) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != r->device) {
      cudaGetLastError();
      return DP_ERR_INVALID_ARG;
    }
  }
  for (int k = 0; k < r->K; ++k)
    if (!grads[k] && r->numel[p]) return DP_ERR_INVALID_ARG;  // an empty parameter may be NULL
  for (int k = 0; k < r->K; ++k) r->grads[(size_t)p * r->K + k] = grads[k];
  r->ready[p] = 1;
  r->pending[r->bucket_of[p]] -= 1;
  int n = 0;
  while (r->next_bucket < (int)r->members.size() && r->pending[r->next_bucket] == 0) {
    dp_status_t st = launch_bucket(r, r->next_bucket, stream);
    if (st != DP_OK) return st;
    ++r->next_bucket;
    ++n;
  }
  if (launched) *launched = n;
  return DP_OK;
}

dp_status_t dp_reducer_finish(dp_reducer_t* r, int* first_pending) {
  if (first_pending) *first_pending = -1;
  if (!r) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(r->mu);
  const bool complete = r->next_bucket == (int)r->members.size();
  if (!complete && first_pending) *first_pending = r->next_bucket;
  reset_iteration(r);
  return complete ? DP_OK : DP_ERR_INVALID_ARG;
}

dp_status_t dp_reducer_set_dry_run(dp_reducer_t* r, int on) {
  if (!r) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(r->mu);
  r->dry_run = on != 0;
  return DP_OK;
}

int dp_reducer_launch_log(dp_reducer_t* r, int* buckets, int cap) {
  if (!r) return 0;
  std::lock_guard<std::mutex> lock(r->mu);
  const int n = (int)r->launch_log.size();
  if (buckets)
    for (int i = 0; i < n && i < cap; ++i) buckets[i] = r->launch_log[i];
  return n;
}

}  // extern "C"
