// Allocation-free variant of mvp_attn_fwd_varlen.
//
// Some callers cannot allocate device memory at the point where they run
// attention: a serving engine that has already handed all free GPU memory to
// its KV-cache pool, a plugin living inside a host framework that owns the
// allocator, or a latency-critical path that must not pay for (or synchronise
// on) an allocation.  Such callers cannot provide the split-KV workspace that
// mvp_attn_fwd_varlen takes.  This entry point uses a fixed scratch array that
// is part of the library's device image instead: every GPU that loads the
// library holds kStaticScratchBytes for it until the process exits.
//
// The scratch is used like a caller's workspace: a header with the prefill
// kernel's work-queue word, then the split-KV partial results (max, sum and
// unnormalised output per split) from the decode kernel to the combine kernel
// of the same call.  The queue word carries a per-launch tag and every
// partial slot the combine reads is written by that call's decode kernel
// (empty splits write a neutral partial), so nothing has to be cleared
// between calls.  All calls share the one array: two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on
// it and may return wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mvp.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
constexpr size_t kHeaderBytes = 256;                 // work-queue header ahead of the partials

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  The name
// g_static_scratch in host code is only a host-side handle, never a device
// address; the address is fetched once per device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t mvp_static_scratch_bytes(void) { return kStaticScratchBytes; }

int mvp_attn_fwd_varlen_static_ws(const void* q, const void* k, const void* v, void* out, float* lse,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                  const int32_t* context_lens, int num_reqs, int total_q, int total_k,
                                  int max_q_len, int max_k_len, int num_decode_reqs, int num_heads_q,
                                  int num_heads_kv, int head_dim, const int32_t* range_table,
                                  const int32_t* range_covered, int causal, int window_left, int window_right,
                                  const float* sinks, int sink_mode, float scale, void* stream) {
  if (num_reqs < 1 || num_decode_reqs < -1 || num_decode_reqs > num_reqs) return MVP_ERR_ARG;
  if (num_heads_q < 1 || head_dim < 1) return MVP_ERR_ARG;
  // The attention call splits long decode rows over as many CTAs as the
  // scratch holds partials for; the array must hold at least one split's
  // partials of the decode rows (the stated maximum batch).
  const size_t decode_reqs = static_cast<size_t>(num_decode_reqs < 0 ? num_reqs : num_decode_reqs);
  const size_t one_split = decode_reqs * static_cast<size_t>(num_heads_q) * (static_cast<size_t>(head_dim) + 2) * 4;
  if (kHeaderBytes + one_split > kStaticScratchBytes) return MVP_ERR_CAPACITY;  // batch too large for the array
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MVP_ERR_CUDA;
  return mvp_attn_fwd_varlen(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, context_lens, num_reqs, total_q,
                             total_k, max_q_len, max_k_len, num_decode_reqs, num_heads_q, num_heads_kv, head_dim,
                             range_table, range_covered, causal, window_left, window_right, sinks, sink_mode,
                             scale, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
