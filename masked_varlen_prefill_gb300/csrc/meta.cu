// Step metadata for CUDA-graph replays: pinned host staging, one
// asynchronous copy into persistent device arrays, and the range-table fill
// on the device.
//
// Restates the persistent-buffer design of vLLM PR #50294 review,
// "Implementation breakdown" step 3 (FlashAttentionMetadataBuilder): the
// builder allocates a pinned host staging area and a device buffer sized for
// the largest batch once, fills the staging area on the host each step from
// the query offsets and the seq_lens upper bound, and copies it to the device
// without blocking.  Here every array of a step (query offsets, key lengths,
// their prefix sums, the fill's upper bounds and the ranges) lives in ONE
// block padded to the capacity (max_reqs requests, max_tokens rows), so that
// a step is exactly one copy of a fixed size plus one fill launch over fixed
// pointers -- the same operations whatever the batch, which is what a
// captured graph replays.  Declarations and contracts are in include/mvp.h.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/mvp.h"
#include "mvp_internal.cuh"

namespace mvp {
namespace {

// Element offsets (int32 units) of the arrays inside a block; the ranges
// start on an 8-byte boundary (the fill reads them as int2).
struct MetaLayout {
  size_t qsl, seq_k, cu_k, bound, ranges, total;
};

MetaLayout meta_layout(int max_reqs, int max_ranges) {
  MetaLayout l;
  const size_t r = static_cast<size_t>(max_reqs);
  l.qsl = 0;
  l.seq_k = l.qsl + r + 1;
  l.cu_k = l.seq_k + r;
  l.bound = l.cu_k + r + 1;
  l.ranges = l.bound + r;
  l.ranges += l.ranges & 1;
  l.total = l.ranges + r * static_cast<size_t>(max_ranges) * 2;
  l.total += l.total & 1;
  return l;
}

bool capacity_ok(int max_reqs, int max_tokens, int max_ranges) {
  return max_reqs >= 1 && max_reqs <= 65535 && max_tokens >= 1 && max_ranges >= 0 && max_ranges <= 4096;
}

}  // namespace
}  // namespace mvp

struct mvp_meta {
  int max_reqs = 0, max_tokens = 0, max_ranges = 0;
  mvp::MetaLayout layout{};
  int32_t* host = nullptr;     // pinned staging block (owned)
  int32_t* dev = nullptr;      // device block (caller's)
  int32_t* table = nullptr;    // device [max_tokens, 2] (caller's)
  int32_t* covered = nullptr;  // device scalar (caller's)
  cudaEvent_t copied = nullptr;
};

extern "C" {

size_t mvp_meta_block_bytes(int max_reqs, int max_ranges) {
  if (max_reqs < 1 || max_reqs > 65535 || max_ranges < 0 || max_ranges > 4096) return 0;
  return mvp::meta_layout(max_reqs, max_ranges).total * sizeof(int32_t);
}

int mvp_meta_offsets(int max_reqs, int max_ranges, size_t* offsets) {
  if (offsets == nullptr || mvp_meta_block_bytes(max_reqs, max_ranges) == 0) return MVP_ERR_ARG;
  const mvp::MetaLayout l = mvp::meta_layout(max_reqs, max_ranges);
  offsets[0] = l.qsl;
  offsets[1] = l.seq_k;
  offsets[2] = l.cu_k;
  offsets[3] = l.bound;
  offsets[4] = l.ranges;
  return MVP_OK;
}

int mvp_meta_pack(const int32_t* query_start_loc, const int32_t* seq_lens_k, const int32_t* seq_lens_bound,
                  const int32_t* ranges, int num_reqs, int num_ranges, int max_reqs, int max_tokens,
                  int max_ranges, int32_t* block) {
  if (!mvp::capacity_ok(max_reqs, max_tokens, max_ranges) || block == nullptr) return MVP_ERR_ARG;
  if (num_reqs < 0 || num_reqs > max_reqs) return MVP_ERR_CAPACITY;
  if (num_ranges < 0 || (ranges != nullptr && num_ranges > max_ranges)) return MVP_ERR_CAPACITY;
  if (num_reqs > 0 && (query_start_loc == nullptr || (seq_lens_k == nullptr && seq_lens_bound == nullptr)))
    return MVP_ERR_ARG;
  const int32_t* bound = seq_lens_bound ? seq_lens_bound : seq_lens_k;
  // validate everything before writing anything
  if (num_reqs > 0 && query_start_loc[0] != 0) return MVP_ERR_ARG;
  long long total_k = 0;
  for (int b = 0; b < num_reqs; ++b) {
    const long long ql = static_cast<long long>(query_start_loc[b + 1]) - query_start_loc[b];
    if (ql < 0) return MVP_ERR_ARG;
    if (seq_lens_k && seq_lens_k[b] < ql) return MVP_ERR_ARG;  // fewer keys than queries
    if (bound[b] < ql) return MVP_ERR_ARG;
    if (seq_lens_k) total_k += seq_lens_k[b];
  }
  if (total_k > INT_MAX) return MVP_ERR_ARG;
  const int num_tokens = num_reqs > 0 ? query_start_loc[num_reqs] : 0;
  if (num_tokens > max_tokens) return MVP_ERR_CAPACITY;

  const mvp::MetaLayout l = mvp::meta_layout(max_reqs, max_ranges);
  int32_t* qsl = block + l.qsl;
  int32_t* sk = block + l.seq_k;
  int32_t* cuk = block + l.cu_k;
  int32_t* bd = block + l.bound;
  int32_t* rg = block + l.ranges;
  // Requests past num_reqs are padding: no rows, no keys, no ranges.
  int32_t acc = 0;
  qsl[0] = 0;
  cuk[0] = 0;
  for (int b = 0; b < max_reqs; ++b) {
    const bool real = b < num_reqs;
    qsl[b + 1] = real ? query_start_loc[b + 1] : num_tokens;
    sk[b] = real && seq_lens_k ? seq_lens_k[b] : 0;
    acc += sk[b];
    cuk[b + 1] = acc;
    bd[b] = real ? bound[b] : 0;
  }
  const size_t per_req = static_cast<size_t>(max_ranges) * 2;
  if (per_req > 0) {
    std::memset(rg, 0, static_cast<size_t>(max_reqs) * per_req * sizeof(int32_t));
    if (ranges != nullptr)
      for (int b = 0; b < num_reqs; ++b)
        std::memcpy(rg + b * per_req, ranges + static_cast<size_t>(b) * num_ranges * 2,
                    static_cast<size_t>(num_ranges) * 2 * sizeof(int32_t));
  }
  for (size_t i = l.ranges + static_cast<size_t>(max_reqs) * per_req; i < l.total; ++i) block[i] = 0;
  for (size_t i = l.bound + max_reqs; i < l.ranges; ++i) block[i] = 0;
  return MVP_OK;
}

int mvp_meta_create(int max_reqs, int max_tokens, int max_ranges, int32_t* device_block, int32_t* range_table,
                    int32_t* range_covered, mvp_meta** out) {
  if (out == nullptr) return MVP_ERR_ARG;
  *out = nullptr;
  if (!mvp::capacity_ok(max_reqs, max_tokens, max_ranges)) return MVP_ERR_ARG;
  if (device_block == nullptr || range_table == nullptr || range_covered == nullptr) return MVP_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(device_block) & 15u) != 0 || (reinterpret_cast<uintptr_t>(range_table) & 7u) != 0)
    return MVP_ERR_UNSUPPORTED;
  mvp_meta* m = new (std::nothrow) mvp_meta;
  if (m == nullptr) return MVP_ERR_CUDA;
  m->max_reqs = max_reqs;
  m->max_tokens = max_tokens;
  m->max_ranges = max_ranges;
  m->layout = mvp::meta_layout(max_reqs, max_ranges);
  m->dev = device_block;
  m->table = range_table;
  m->covered = range_covered;
  void* h = nullptr;
  if (cudaHostAlloc(&h, m->layout.total * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess) {
    delete m;
    return MVP_ERR_CUDA;
  }
  m->host = static_cast<int32_t*>(h);
  // An empty batch until the first stage.
  mvp_meta_pack(nullptr, nullptr, nullptr, nullptr, 0, 0, max_reqs, max_tokens, max_ranges, m->host);
  if (cudaEventCreateWithFlags(&m->copied, cudaEventDisableTiming) != cudaSuccess) {
    cudaFreeHost(m->host);
    delete m;
    return MVP_ERR_CUDA;
  }
  *out = m;
  return MVP_OK;
}

int mvp_meta_destroy(mvp_meta* m) {
  if (m == nullptr) return MVP_OK;
  int rc = MVP_OK;
  if (m->copied && cudaEventSynchronize(m->copied) != cudaSuccess) rc = MVP_ERR_CUDA;
  if (m->copied) cudaEventDestroy(m->copied);
  if (m->host) cudaFreeHost(m->host);
  delete m;
  return rc;
}

int mvp_meta_stage(mvp_meta* m, const int32_t* query_start_loc, const int32_t* seq_lens_k,
                   const int32_t* seq_lens_bound, const int32_t* ranges, int num_reqs, int num_ranges) {
  if (m == nullptr) return MVP_ERR_ARG;
  // The staging block is read by the last upload's copy: wait until it ran.
  if (cudaEventSynchronize(m->copied) != cudaSuccess) return MVP_ERR_CUDA;
  return mvp_meta_pack(query_start_loc, seq_lens_k, seq_lens_bound, ranges, num_reqs, num_ranges, m->max_reqs,
                       m->max_tokens, m->max_ranges, m->host);
}

int mvp_meta_upload(mvp_meta* m, void* stream) {
  if (m == nullptr) return MVP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(m->dev, m->host, m->layout.total * sizeof(int32_t), cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return MVP_ERR_CUDA;
  // Inside a capture the record becomes a node of the graph, so that every
  // replay marks the staging block free again.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MVP_ERR_CUDA;
  const cudaError_t e = cs == cudaStreamCaptureStatusActive
                            ? cudaEventRecordWithFlags(m->copied, st, cudaEventRecordExternal)
                            : cudaEventRecord(m->copied, st);
  if (e != cudaSuccess) return MVP_ERR_CUDA;
  mvp::FillParams p;
  p.ranges = m->max_ranges > 0 ? m->dev + m->layout.ranges : nullptr;
  p.qsl = m->dev + m->layout.qsl;
  p.seq_lens = m->dev + m->layout.bound;
  p.out = m->table;
  p.rows_written = m->covered;
  p.num_reqs = m->max_reqs;
  p.max_ranges = m->max_ranges;
  p.num_tokens = m->max_tokens;
  if (mvp::launch_fill(p, st) != cudaSuccess) return MVP_ERR_CUDA;
  return MVP_OK;
}

}  // extern "C"
