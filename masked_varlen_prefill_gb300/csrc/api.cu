// C-ABI host layer: argument validation, TMA tensor-map encoding, launch
// planning.  Declarations and argument contracts are in include/mvp.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mvp.h"
#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {
namespace {

// One error word per device, living in this module's device memory: kernels
// write a timeout code there (ptx.cuh), mvp_get_last_device_error reads it.
__device__ int g_device_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
thread_local int g_last_launches = 0;

// The second stream of a device on which the decode kernel of a mixed batch
// runs beside the prefill kernel, and the events that fork it from and join
// it back to the caller's stream.  Created with the rest of the per-device
// state on the first attention call on the device and kept for the life of
// the process.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
  std::mutex mutex;  // one fork / launch / join sequence at a time
};
SideStream g_side[kMaxDevices];

cudaError_t device_state(int** err_ptr, int* num_sms = nullptr, SideStream** side = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error_word);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<int*>(ptr);
  }
  if (g_num_sms[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = n > 0 ? n : 1;
  }
  SideStream& ss = g_side[dev];
  if (ss.stream == nullptr) {
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if ((e = cudaEventCreateWithFlags(&f, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&j, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking)) != cudaSuccess) return e;
    ss.fork = f;
    ss.join = j;
    ss.stream = st;
  }
  *err_ptr = g_err_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  if (side) *side = &ss;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D bf16 tensor [rows, heads, dim] (dim innermost) -> tiled TMA map.
bool encode_3d(CUtensorMap* map, const void* base, int dim, int heads, int rows, int box_x, int box_y,
               int box_z, bool swizzle128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dim) * 2, static_cast<cuuint64_t>(heads) * dim * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y),
                       static_cast<cuuint32_t>(box_z)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int largest_pow2_divisor(int g, int cap) {
  int p = 1;
  while (p * 2 <= cap && g % (p * 2) == 0) p *= 2;
  return p;
}

constexpr int kDecodeChunk = 4096;
constexpr int kMaxSplits = 64;

}  // namespace
}  // namespace mvp

using namespace mvp;

extern "C" {

const char* mvp_status_str(int status) {
  switch (status) {
    case MVP_OK: return "ok";
    case MVP_ERR_ARG: return "invalid argument";
    case MVP_ERR_CAPACITY: return "output capacity too small";
    case MVP_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case MVP_ERR_CUDA: return "CUDA error";
    case MVP_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MVP_ERR_DEVICE_BOUNDS: return "device-side index out of bounds (bounds-checked build)";
    default: return "unknown status";
  }
}

int mvp_last_launch_count(void) { return g_last_launches; }

int mvp_fill_query_ranges(const int32_t* ranges, int num_reqs, int max_ranges, const int32_t* query_start_loc,
                          const int32_t* seq_lens, int num_tokens, int32_t* out, int out_capacity,
                          int32_t* rows_written, void* stream) {
  g_last_launches = 0;
  if (num_reqs < 0 || max_ranges < 0 || num_tokens < 0 || out_capacity < 0) return MVP_ERR_ARG;
  if (num_tokens > 0) {
    if (num_reqs < 1 || query_start_loc == nullptr || seq_lens == nullptr || out == nullptr) return MVP_ERR_ARG;
    if (max_ranges > 0 && ranges == nullptr) return MVP_ERR_ARG;
    if (num_tokens > out_capacity) return MVP_ERR_CAPACITY;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return MVP_ERR_UNSUPPORTED;
    if (ranges != nullptr && (reinterpret_cast<uintptr_t>(ranges) & 7u) != 0) return MVP_ERR_UNSUPPORTED;
  }
  FillParams p;
  p.ranges = ranges;
  p.qsl = query_start_loc;
  p.seq_lens = seq_lens;
  p.out = out;
  p.rows_written = rows_written;
  p.num_reqs = num_reqs;
  p.max_ranges = ranges ? max_ranges : 0;
  p.num_tokens = num_tokens;
  cudaError_t e = launch_fill(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return MVP_ERR_CUDA;
  g_last_launches = num_tokens > 0 ? 1 : 0;  // kernels only (the flag reset is a memset)
  return MVP_OK;
}

size_t mvp_attn_workspace_size(int num_reqs, int num_heads_q, int head_dim, int max_k_len) {
  if (num_reqs < 0 || num_heads_q <= 0 || head_dim <= 0 || max_k_len <= 0) return 0;
  int splits = (max_k_len + kDecodeChunk - 1) / kDecodeChunk;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits < 2 || num_reqs == 0) return mvp::kWorkspaceHeader;
  return mvp::kWorkspaceHeader + static_cast<size_t>(num_reqs) * num_heads_q * splits * (head_dim + 2) * sizeof(float);
}

}  // extern "C"

namespace mvp {
namespace {

// Where the keys and values live: packed ([total_k, Hkv, D] with row offsets
// cu_k) or paged ([num_blocks * block_size, Hkv, D] addressed through a
// block table, keys per request in seq_k).
struct KVArgs {
  const void* k;
  const void* v;
  long long rows;  // rows of the K/V tensors
  const int32_t* cu_k;
  const int32_t* seq_k;
  const int32_t* block_table;
  int block_shift;
  int max_blocks;
};

// SMs for the prefill kernel of a mixed batch while the decode kernel runs
// beside it, or 0 to run the two one after the other.  The decode kernel's
// rate grows with its SMs up to the HBM peak (measured on the decode rows of
// the mixed serving batches: ~53 GB/s per SM, 5.5 TB/s on 104 SMs), and its
// CTAs spread over the prefill kernel's SMs once that finishes; the prefill
// kernel's persistent grid is fixed at launch, so a share too small makes the
// prefill side the long pole (5b: 0.98 ms at 32 SMs against 0.78 at 48),
// while a share too large only delays the decode rows a little (0.83 ms at
// 96).  The share is the prefill side's part of the two sides' estimated
// work, 1.2 times over (the measured optimum: 24 and 48 SMs for the two
// serving batches, whose prefill sides are 13 and 26 % of the work), at
// most three quarters of the SMs; it overlaps only when the decode side's
// estimated time (K/V bytes at the HBM rate) is at least a third of the
// prefill side's (FLOPs at the tensor rate).  The key counts are device
// data, so the estimates use an average key run per request (total_k /
// num_reqs packed, max_k_len paged) capped by the window.  A paged cache of
// blocks under 64 tokens loads the prefill kernel's tiles in as many boxes
// as blocks, which slows it (mm_prefix sliding: 0.39 of the bf16 peak at 16
// tokens against 0.65 at 64 and packed), so its rate estimate shrinks with
// the block: x0.6 at 16 tokens, x0.8 at 32.
constexpr double kDecodeBytesPerS = 6.0e12;
constexpr double kPrefillFlopsPerS = 1.1e15;

int mixed_prefill_sms(int num_sms, int total_q, int total_k, bool paged, int block_shift, int num_reqs,
                      int decode_rows, int max_q_len, int max_k_len, int causal, int window_left, int window_right,
                      int hq, int hkv) {
  const double avg_k = paged ? static_cast<double>(max_k_len) : static_cast<double>(total_k) / num_reqs;
  double span = avg_k;  // keys one row sees
  if (causal) {
    if (window_left >= 0) span = std::min(span, window_left + 1.0);
  } else if (window_left >= 0 && window_right >= 0) {
    span = std::min(span, window_left + window_right + 1.0);
  }
  const double pre_rows = std::max(0, total_q - decode_rows);
  const double pre_span = causal && window_left < 0 ? std::max(1.0, avg_k - 0.5 * max_q_len) : span;
  const double t_dec = 4.0 * hkv * decode_rows * span / kDecodeBytesPerS;    // per unit of head_dim
  const double box_rate = (paged && block_shift < 6) ? std::max(0.2, 0.6 + 0.2 * (block_shift - 4)) : 1.0;
  const double t_pre = 4.0 * hq * pre_rows * pre_span / (kPrefillFlopsPerS * box_rate);  // per unit of head_dim
  if (t_dec * 3.0 < t_pre) return 0;
  const int cap = (3 * num_sms) / 4;
  int sms = static_cast<int>(std::ceil(1.2 * num_sms * t_pre / (t_pre + t_dec)));
  sms = std::max(2, std::min(sms + (sms & 1), cap - (cap & 1)));  // whole CTA pairs
  return sms;
}

int attn_fwd_impl(const void* q, void* out, float* lse, const int32_t* cu_seqlens_q, const int32_t* context_lens,
                  int num_reqs, int total_q, int max_q_len, int max_k_len, int num_decode_reqs, int num_heads_q,
                  int num_heads_kv, int head_dim, const int32_t* range_table, const int32_t* range_covered,
                  int causal, int window_left, int window_right, const float* sinks, int sink_mode, float scale,
                  void* workspace, size_t workspace_bytes, void* stream, const KVArgs& kv,
                  const int32_t* scan_ranges = nullptr, int max_ranges = 0,
                  const mvp_attn_options* opts = nullptr) {
  const void* k = kv.k;
  const void* v = kv.v;
  const bool paged = kv.block_table != nullptr;
  // ------------------------------------------------------------ validation
  if (num_reqs < 1 || num_reqs > 65535 || total_q < 0 || kv.rows < 0) return MVP_ERR_ARG;
  if (num_heads_q < 1 || num_heads_kv < 1 || num_heads_q % num_heads_kv != 0) return MVP_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256 && head_dim != 512) return MVP_ERR_UNSUPPORTED;
  if (sink_mode < 0 || sink_mode > 2) return MVP_ERR_ARG;
  if (sink_mode != 0 && sinks == nullptr) return MVP_ERR_ARG;
  if (window_left < -1 || window_right < -1) return MVP_ERR_ARG;
  if (causal != 0 && causal != 1) return MVP_ERR_ARG;
  if (num_decode_reqs < -1 || num_decode_reqs > num_reqs) return MVP_ERR_ARG;
  if (!(scale > 0.f) || scale > 3.0e38f) return MVP_ERR_ARG;  // NaN, <= 0, inf
  if (total_q == 0) return MVP_OK;
  if (kv.rows < 1 || kv.rows > INT_MAX || max_q_len < 1 || max_k_len < 1) return MVP_ERR_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || cu_seqlens_q == nullptr ||
      (paged ? kv.seq_k == nullptr : kv.cu_k == nullptr))
    return MVP_ERR_ARG;
  const int total_k = static_cast<int>(kv.rows);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return MVP_ERR_UNSUPPORTED;
  if (range_table != nullptr && (reinterpret_cast<uintptr_t>(range_table) & 7u) != 0) return MVP_ERR_UNSUPPORTED;
  if (max_ranges < 0 || max_ranges > 4096 || (max_ranges > 0 && scan_ranges == nullptr)) return MVP_ERR_ARG;
  if (max_ranges == 0) scan_ranges = nullptr;
  if (scan_ranges != nullptr && range_table != nullptr) return MVP_ERR_ARG;
  if (scan_ranges != nullptr && (reinterpret_cast<uintptr_t>(scan_ranges) & 7u) != 0) return MVP_ERR_UNSUPPORTED;
  if (static_cast<long long>(total_q) * num_heads_q * head_dim >= (1LL << 40)) return MVP_ERR_UNSUPPORTED;
  if (opts != nullptr) {
    if (opts->variant != MVP_VARIANT_DEFAULT && opts->variant != MVP_VARIANT_D512_HEAD_SPLIT) return MVP_ERR_ARG;
    if (opts->variant == MVP_VARIANT_D512_HEAD_SPLIT && head_dim != 512) return MVP_ERR_UNSUPPORTED;
    if (opts->fault != MVP_FAULT_NONE && opts->fault != MVP_FAULT_WITHHOLD_PROBS) return MVP_ERR_ARG;
  }
  const bool d512_split = opts != nullptr && opts->variant == MVP_VARIANT_D512_HEAD_SPLIT;

  // Paged: a TMA box never crosses a cache block.
  auto box_rows = [&](int rows) { return paged ? (rows < (1 << kv.block_shift) ? rows : (1 << kv.block_shift)) : rows; };
  int* err = nullptr;
  int num_sms = 1;
  SideStream* side = nullptr;
  if (device_state(&err, &num_sms, &side) != cudaSuccess) return MVP_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  MaskParams m;
  m.cu_q = cu_seqlens_q;
  m.cu_k = paged ? nullptr : kv.cu_k;
  m.seq_k = paged ? kv.seq_k : nullptr;
  m.block_table = kv.block_table;
  m.block_shift = paged ? kv.block_shift : 0;
  m.max_blocks = paged ? kv.max_blocks : 0;
  m.ctx_lens = context_lens;
  m.table = range_table;
  m.covered = range_table ? range_covered : nullptr;
  m.ranges = scan_ranges;
  m.max_ranges = scan_ranges ? max_ranges : 0;
  m.sinks = sink_mode ? sinks : nullptr;
  m.causal = causal;
  m.window_left = window_left;
  m.window_right = causal ? 0 : window_right;
  m.sink_mode = sink_mode;
  m.scale_log2 = scale * 1.4426950408889634f;
  m.scale = scale;
  m.wait_limit_us = (opts != nullptr && opts->wait_limit_us != 0) ? opts->wait_limit_us : kDefaultWaitLimitUs;
  m.fault = opts != nullptr ? opts->fault : kFaultNone;
  m.total_q = total_q;
  m.err = err;

  const int group = num_heads_q / num_heads_kv;
  int launches = 0;
  // Workspace: the prefill work-queue word in its header, the decode split
  // partials after it.  Without a usable header, static scheduling and no
  // split.
  unsigned long long* queue = nullptr;
  void* partials = nullptr;
  size_t partial_bytes = 0;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 15u) == 0 &&
      workspace_bytes >= kWorkspaceHeader) {
    queue = static_cast<unsigned long long*>(workspace);
    partials = static_cast<unsigned char*>(workspace) + kWorkspaceHeader;
    partial_bytes = workspace_bytes - kWorkspaceHeader;
  }

  const int prefill_first = num_decode_reqs < 0 ? 0 : num_decode_reqs;
  const int decode_count = num_decode_reqs < 0 ? num_reqs : num_decode_reqs;

  // ------------------------------------------------------------ prefill rows
  const bool run_prefill = max_q_len > 1 && prefill_first < num_reqs;
  PrefillParams pp{};
  CUtensorMap pmq, pmk, pmv;
  if (run_prefill) {
    const PrefillShape shape = prefill_tile_shape(head_dim, d512_split);
    const int gpack = largest_pow2_divisor(group, 8);
    const int bmp = 128 / gpack;
    pp.m = m;
    pp.out = out;
    pp.lse = lse;
    pp.err = err;
    pp.num_reqs = num_reqs;
    pp.total_q = total_q;
    pp.hq = num_heads_q;
    pp.hkv = num_heads_kv;
    pp.gpack = gpack;
    pp.n_hgroups = group / gpack;
    const int item_pos = shape.item_rows / gpack;  // query positions per work item
    pp.n_qtiles = (max_q_len + item_pos - 1) / item_pos;
    pp.skip_decode = 1;
    pp.req_offset = prefill_first;
    pp.n_ctas = num_sms;
    // The work queue evens out items of very different cost, which is what
    // an unwindowed mask makes (an item's keys grow with its position and
    // context) and what range lists make under a window (a bidirectional
    // range extends only the items whose rows it holds).  Under a window
    // without ranges every item's keys are capped at the window, the static
    // stride is already even, and the queued round measured slower (mixed
    // batch with a 4096 window: 50 vs 52 % of peak); with ranges it measured
    // faster (mm-prefix sliding window: 62.4 vs 61.3 %, chunked prefill:
    // 90.6 vs 89.4 %).
    const bool ranged = range_table != nullptr || scan_ranges != nullptr;
    pp.queue = (window_left < 0 || window_left >= max_k_len || ranged) ? queue : nullptr;
    if (!encode_3d(&pmq, q, head_dim, num_heads_q, total_q, 64, gpack, bmp, true) ||
        !encode_3d(&pmk, k, head_dim, num_heads_kv, total_k, 64, 1, box_rows(shape.k_box_keys), true) ||
        !encode_3d(&pmv, v, head_dim, num_heads_kv, total_k, 64, 1, box_rows(shape.v_box_keys), true))
      return MVP_ERR_UNSUPPORTED;
  }

  // ------------------------------------------------------------ decode rows
  const bool run_decode = decode_count > 0;
  DecodeParams dp{};
  CUtensorMap dmk, dmv;
  if (run_decode) {
    dp.m = m;
    dp.q = q;
    dp.out = out;
    dp.lse = lse;
    dp.err = err;
    dp.num_reqs = decode_count;
    dp.total_q = total_q;
    dp.hq = num_heads_q;
    dp.hkv = num_heads_kv;
    dp.group = group;
    const int kt = decode_keys_per_tile(head_dim);
    // Keys a decode row's CTA walks: its visible hull, started on a multiple
    // of the tile size (the kernel aligns it down by up to kt - 1 keys).
    long long span = max_k_len;
    if (causal && window_left >= 0 && range_table == nullptr && scan_ranges == nullptr && context_lens == nullptr)
      span = (window_left + static_cast<long long>(kt) < span) ? window_left + static_cast<long long>(kt) : span;
    int splits = static_cast<int>((span + kDecodeChunk - 1) / kDecodeChunk);
    if (splits > kMaxSplits) splits = kMaxSplits;
    const size_t per_split = static_cast<size_t>(decode_count) * num_heads_q * (head_dim + 2) * sizeof(float);
    if (partials == nullptr) splits = 1;
    else if (static_cast<size_t>(splits) * per_split > partial_bytes)
      splits = static_cast<int>(partial_bytes / per_split);
    if (splits < 2) splits = 1;
    long long chunk = (span + splits - 1) / splits;
    chunk = ((chunk + kt - 1) / kt) * kt;
    if (chunk > INT_MAX) chunk = INT_MAX;
    dp.n_splits = splits;
    dp.chunk = static_cast<int>(chunk);
    dp.partial = splits > 1 ? static_cast<float*>(partials) : nullptr;
    const int per_cta = decode_heads_per_cta(head_dim, group);
    if (static_cast<long long>(num_heads_kv) * ((group + per_cta - 1) / per_cta) > 65535) return MVP_ERR_UNSUPPORTED;
    const int box = decode_box_inner(head_dim);
    if (!encode_3d(&dmk, k, head_dim, num_heads_kv, total_k, box, 1, box_rows(kt), false) ||
        !encode_3d(&dmv, v, head_dim, num_heads_kv, total_k, box, 1, box_rows(kt), false))
      return MVP_ERR_UNSUPPORTED;
  }

  // ------------------------------------------------------------ launches
  // Both kernels: the decode kernel (HBM-bound) may run beside the prefill
  // kernel (tensor-bound) instead of after it.  The prefill kernel's
  // persistent CTAs then take a share of the SMs (mixed_prefill_sms) and the
  // decode kernel goes to the device's side stream, forked from and joined
  // back to the caller's stream with events (capturable in a CUDA graph).
  // The decode-first order (num_decode_reqs >= 0) is required: it tells how
  // many rows each side has.
  const int share = (opts != nullptr) ? opts->mixed_prefill_sms : 0;
  bool concurrent = run_prefill && run_decode && num_decode_reqs >= 0 && share >= 0 && num_sms >= 4;
  int sms = 0;
  if (concurrent) {
    sms = share > 0 ? share
                    : mixed_prefill_sms(num_sms, total_q, total_k, paged, paged ? kv.block_shift : 0, num_reqs,
                                        decode_count, max_q_len, max_k_len, causal, window_left, window_right,
                                        num_heads_q, num_heads_kv);
    if (sms == 0) concurrent = false;               // too little decode work to overlap
    if (sms > num_sms - 2) sms = num_sms - 2;       // leave the decode kernel at least two SMs
    if (sms < 2) sms = 2;
  }
  if (!concurrent) {
    if (run_prefill) {
      if (launch_prefill(head_dim, d512_split, pp, pmq, pmk, pmv, st) != cudaSuccess) return MVP_ERR_CUDA;
      ++launches;
    }
    if (run_decode && launch_decode(head_dim, dp, dmk, dmv, st, &launches) != cudaSuccess) return MVP_ERR_CUDA;
  } else {
    pp.n_ctas = sms;
    std::lock_guard<std::mutex> lock(side->mutex);  // one fork / join at a time per device
    if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
      return MVP_ERR_CUDA;
    if (launch_prefill(head_dim, d512_split, pp, pmq, pmk, pmv, st) != cudaSuccess) return MVP_ERR_CUDA;
    ++launches;
    if (launch_decode(head_dim, dp, dmk, dmv, side->stream, &launches) != cudaSuccess) return MVP_ERR_CUDA;
    if (cudaEventRecord(side->join, side->stream) != cudaSuccess || cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess)
      return MVP_ERR_CUDA;
  }
  g_last_launches = launches;
  return MVP_OK;
}

}  // namespace
}  // namespace mvp

extern "C" {

int mvp_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* context_lens,
                        int num_reqs, int total_q, int total_k, int max_q_len, int max_k_len, int num_decode_reqs,
                        int num_heads_q, int num_heads_kv, int head_dim, const int32_t* range_table,
                        const int32_t* range_covered, int causal, int window_left, int window_right,
                        const float* sinks, int sink_mode, float scale, void* workspace, size_t workspace_bytes,
                        void* stream) {
  g_last_launches = 0;
  KVArgs kv{k, v, total_k, cu_seqlens_k, nullptr, nullptr, 0, 0};
  return attn_fwd_impl(q, out, lse, cu_seqlens_q, context_lens, num_reqs, total_q, max_q_len, max_k_len,
                       num_decode_reqs, num_heads_q, num_heads_kv, head_dim, range_table, range_covered, causal,
                       window_left, window_right, sinks, sink_mode, scale, workspace, workspace_bytes, stream, kv);
}

int mvp_attn_fwd_varlen_ext(const void* q, const void* k, const void* v, void* out, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* context_lens,
                            int num_reqs, int total_q, int total_k, int max_q_len, int max_k_len,
                            int num_decode_reqs, int num_heads_q, int num_heads_kv, int head_dim,
                            const int32_t* range_table, const int32_t* range_covered, int causal, int window_left,
                            int window_right, const float* sinks, int sink_mode, float scale, void* workspace,
                            size_t workspace_bytes, void* stream, const mvp_attn_options* options) {
  g_last_launches = 0;
  KVArgs kv{k, v, total_k, cu_seqlens_k, nullptr, nullptr, 0, 0};
  return attn_fwd_impl(q, out, lse, cu_seqlens_q, context_lens, num_reqs, total_q, max_q_len, max_k_len,
                       num_decode_reqs, num_heads_q, num_heads_kv, head_dim, range_table, range_covered, causal,
                       window_left, window_right, sinks, sink_mode, scale, workspace, workspace_bytes, stream, kv,
                       nullptr, 0, options);
}

int mvp_attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, const int32_t* block_table,
                       int block_size, int max_blocks_per_seq, int num_blocks, const int32_t* context_lens,
                       int num_reqs, int total_q, int max_q_len, int max_k_len, int num_decode_reqs, int num_heads_q,
                       int num_heads_kv, int head_dim, const int32_t* range_table, const int32_t* range_covered,
                       int causal, int window_left, int window_right, const float* sinks, int sink_mode, float scale,
                       void* workspace, size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  int shift = 0;
  while (shift < 30 && (1 << shift) < block_size) ++shift;
  if (block_size < 16 || block_size > 256 || (1 << shift) != block_size) return MVP_ERR_ARG;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || block_table == nullptr || seq_lens_k == nullptr)
    return MVP_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * block_size < max_k_len) return MVP_ERR_ARG;
  if (static_cast<long long>(num_blocks) * block_size > INT_MAX) return MVP_ERR_UNSUPPORTED;
  KVArgs kv{k_cache, v_cache, static_cast<long long>(num_blocks) * block_size, nullptr, seq_lens_k, block_table,
            shift, max_blocks_per_seq};
  return attn_fwd_impl(q, out, lse, cu_seqlens_q, context_lens, num_reqs, total_q, max_q_len, max_k_len,
                       num_decode_reqs, num_heads_q, num_heads_kv, head_dim, range_table, range_covered, causal,
                       window_left, window_right, sinks, sink_mode, scale, workspace, workspace_bytes, stream, kv);
}

int mvp_attn_fwd_varlen_scan(const void* q, const void* k, const void* v, void* out, float* lse,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* context_lens,
                             int num_reqs, int total_q, int total_k, int max_q_len, int max_k_len,
                             int num_decode_reqs, int num_heads_q, int num_heads_kv, int head_dim,
                             const int32_t* ranges, int max_ranges, int causal, int window_left, int window_right,
                             const float* sinks, int sink_mode, float scale, void* workspace,
                             size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  KVArgs kv{k, v, total_k, cu_seqlens_k, nullptr, nullptr, 0, 0};
  return attn_fwd_impl(q, out, lse, cu_seqlens_q, context_lens, num_reqs, total_q, max_q_len, max_k_len,
                       num_decode_reqs, num_heads_q, num_heads_kv, head_dim, nullptr, nullptr, causal, window_left,
                       window_right, sinks, sink_mode, scale, workspace, workspace_bytes, stream, kv, ranges,
                       max_ranges);
}

int mvp_get_last_device_error(void* stream) {
  int* err = nullptr;
  if (device_state(&err) != cudaSuccess) return MVP_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MVP_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MVP_ERR_CUDA;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MVP_ERR_CUDA;
    return value == kDevBounds ? MVP_ERR_DEVICE_BOUNDS : MVP_ERR_DEVICE_TIMEOUT;
  }
  return MVP_OK;
}

}  // extern "C"
