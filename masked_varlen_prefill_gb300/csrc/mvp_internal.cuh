// Internal launch interfaces shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mvp {

// ----------------------------------------------------------------- fill
struct FillParams {
  const int32_t* ranges;    // [num_reqs, max_ranges, 2]
  const int32_t* qsl;       // [num_reqs + 1]
  const int32_t* seq_lens;  // [num_reqs]
  int32_t* out;             // [num_tokens, 2]
  int32_t* rows_written;    // device scalar or null
  int num_reqs;
  int max_ranges;
  int num_tokens;
};

cudaError_t launch_fill(const FillParams& p, cudaStream_t stream);

// Faults a caller can ask for to test the bounded-wait path (never set by
// the plain entry points).  kFaultWithholdProbs: the first softmax warp of
// every prefill CTA (rank 0 of each pair) does not signal that its first key
// tile's probabilities are in TMEM, so the MMA issuer's wait for them runs out.
enum FaultInjection : int { kFaultNone = 0, kFaultWithholdProbs = 1 };

// ----------------------------------------------------------------- masks
// Per-row visible set = base interval U range interval (closed, in key
// coordinates of the request).  Shared by the prefill and decode kernels.
struct MaskParams {
  const int32_t* cu_q;
  const int32_t* cu_k;       // packed K/V: [num_reqs + 1] row offsets (null when paged)
  const int32_t* seq_k;      // paged K/V: keys per request [num_reqs] (null when packed)
  const int32_t* block_table;  // paged K/V: [num_reqs, max_blocks] block ids (null when packed)
  int block_shift;           // log2(block size) when paged
  int max_blocks;            // row stride of block_table
  const int32_t* ctx_lens;   // or null
  const int32_t* table;      // [total_q, 2] or null
  const int32_t* covered;    // device scalar or null
  const int32_t* ranges;     // scan mode: [num_reqs, max_ranges, 2] or null (then table is null)
  int max_ranges;
  const float* sinks;        // [hq] or null
  int causal;
  int window_left;           // -1 = unbounded
  int window_right;          // -1 = unbounded (non-causal only)
  int sink_mode;
  float scale_log2;          // scale * log2(e)
  float scale;               // > 0
  uint32_t wait_limit_us;    // budget of one bounded device wait
  int fault;                 // FaultInjection: kFaultNone except in the timeout tests
  // bounds-checked build: rows of q / out / table, and the error word
  int total_q;
  int* err;
};

// ----------------------------------------------------------------- prefill
// Caller workspace layout: this many bytes of header (the prefill kernel's
// work-queue word at offset 0), then the decode kernel's split partials.
constexpr size_t kWorkspaceHeader = 256;

struct PrefillParams {
  MaskParams m;
  void* out;          // bf16 [total_q, hq, D]
  float* lse;         // [hq, total_q] or null
  int* err;           // device error word
  int num_reqs;
  int total_q;
  int hq;
  int hkv;
  int gpack;          // q heads packed into one 128-row tile (power of two)
  int n_hgroups;      // (hq / hkv) / gpack
  int n_qtiles;       // items per (request, head group): ceil(max_q_len / (ncta * 128 / gpack))
  int skip_decode;    // requests with q_len == 1 are left to the decode kernel
  int req_offset;     // first request covered (items walk [req_offset, num_reqs))
  int n_ctas;         // persistent CTAs to launch (SM count)
  unsigned long long* queue;  // work-queue word (caller's workspace), or null: static stride
};

// head_dim in {64, 128, 256, 512}.  Tensor maps are encoded by the caller
// (see api.cu) for the tile shapes prefill_tile_shape() reports.
struct PrefillShape {
  int bn;        // keys per tile
  int dv_cta;    // value columns per CTA
  int dv_split;  // CTAs per (q tile, head group) along the value dimension
  int v_box_keys;  // keys per V TMA box
  int k_box_keys;  // keys per K TMA box (a CTA pair's CTA loads half a tile)
  int ncta;        // CTAs of a cluster working on one item: 1 or 2
  int item_rows;   // query rows (position x head) of one item
  int issuers;     // CTAs of an item that issue MMAs (2 for a head-dim split)
  int qk_k;        // head dims one issuing CTA multiplies in QK
  int oc;          // O columns one issuing CTA accumulates
  int mma_m;       // M of each MMA
  int rowsum_n;    // PV MMA columns that sum the rows (P x ones), 0 when the softmax sums them
};
// d512_head_split selects the head-dim-split form of D = 512 (TMEM-resident
// O, no recomputed QK) instead of the default value split.
PrefillShape prefill_tile_shape(int head_dim, bool d512_head_split);

cudaError_t launch_prefill(int head_dim, bool d512_head_split, const PrefillParams& p, const CUtensorMap& map_q,
                           const CUtensorMap& map_k, const CUtensorMap& map_v, cudaStream_t stream);

// ----------------------------------------------------------------- decode
struct DecodeParams {
  MaskParams m;
  const void* q;        // bf16 [total_q, hq, D]
  void* out;            // bf16 [total_q, hq, D]
  float* lse;           // [hq, total_q] or null
  float* partial;       // [num_reqs, hq, n_splits, D + 2] or null (single split)
  int* err;
  int num_reqs;         // requests covered by the decode grid: [0, num_reqs)
  int total_q;
  int hq;
  int hkv;
  int group;            // hq / hkv
  int n_splits;
  int chunk;            // keys per split
};

cudaError_t launch_decode(int head_dim, const DecodeParams& p, const CUtensorMap& map_k,
                          const CUtensorMap& map_v, cudaStream_t stream, int* launches);
int decode_keys_per_tile(int head_dim);
int decode_box_inner(int head_dim);
// Heads one decode CTA handles for a GQA group of `group` query heads.
inline int decode_heads_per_cta(int head_dim, int group) {
  if (group == 1) return 1;
  if (group == 2) return 2;
  if (group <= 4 || head_dim >= 512) return 4;
  return 8;
}

}  // namespace mvp
