// Per-query-row visibility as two closed key intervals.
//
// For a query at absolute position p of a request with k_len keys:
//   base  = keys allowed by the causal / sliding-window rule
//           (step14_4 tutorial: j > p is masked when causal; vLLM PR #50294
//           mask_mod: the window keeps j >= p - window_left; PR #49815: a
//           symmetric window also keeps j <= p + window_right)
//   range = the row's closed [start, end] from the range table, clamped on
//           the past side by the same window (PR #50294 mask_mod)
// visible = base OR range.  When the table row comes from the fill (its range
// holds p), the two intervals touch at p, so the union is one interval; an
// arbitrary caller table may give two disjoint intervals, which the per-key
// test below still handles exactly.
#pragma once

#include <climits>
#include <cstdint>

#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {

struct RowVis {
  int b_lo, b_hi;  // base interval (empty when b_lo > b_hi)
  int r_lo, r_hi;  // range interval (empty when r_lo > r_hi)

  __device__ __forceinline__ bool visible(int j) const {
    return (j >= b_lo && j <= b_hi) || (j >= r_lo && j <= r_hi);
  }
  __device__ __forceinline__ bool base_empty() const { return b_lo > b_hi; }
  __device__ __forceinline__ bool range_empty() const { return r_lo > r_hi; }
  // Smallest interval holding every visible key (empty: lo > hi).
  __device__ __forceinline__ void hull(int& lo, int& hi) const {
    lo = INT_MAX;
    hi = INT_MIN;
    if (!base_empty()) { lo = b_lo; hi = b_hi; }
    if (!range_empty()) { lo = min(lo, r_lo); hi = max(hi, r_hi); }
  }
  // An interval of keys that are ALL visible (conservative when the two
  // intervals are disjoint: then only the base interval is reported).
  __device__ __forceinline__ void core(int& lo, int& hi) const {
    const bool be = base_empty(), re = range_empty();
    if (be && re) { lo = INT_MAX; hi = INT_MIN; return; }
    if (be) { lo = r_lo; hi = r_hi; return; }
    if (re) { lo = b_lo; hi = b_hi; return; }
    if (r_lo <= b_hi + 1 && b_lo <= r_hi + 1) { lo = min(b_lo, r_lo); hi = max(b_hi, r_hi); return; }
    lo = b_lo;
    hi = b_hi;
  }
};

// Bit i set iff key c0 + i (i < 32) lies in the closed interval [lo, hi].
__device__ __forceinline__ uint32_t interval_bits(int lo, int hi, int c0) {
  const int a = max(lo, c0), b = min(hi, c0 + 31);
  if (a > b) return 0u;
  const uint32_t width = static_cast<uint32_t>(b - a + 1);  // 1..32
  const uint32_t ones = (width >= 32u) ? 0xffffffffu : ((1u << width) - 1u);
  return ones << (a - c0);
}

__device__ __forceinline__ RowVis empty_row() {
  RowVis v;
  v.b_lo = 1; v.b_hi = 0; v.r_lo = 1; v.r_hi = 0;
  return v;
}

// The same from an already loaded table entry (use_range false: range off).
__device__ __forceinline__ RowVis row_visibility_from(const MaskParams& m, int p, int k_len, bool use_range, int2 e);

// Scan mode (the per-request range list of vLLM's Triton path, PR #50294
// "Implementation breakdown" 2): a key is in range iff some valid range
// (start < end) holds both the query position p and the key.  Every range
// that holds p contains p, so their union is one interval: [min start,
// max end] over those ranges, or (-1, -1) when none holds p.  With
// non-overlapping ranges (the page's invariant) it is the table row.
__device__ __forceinline__ int2 scan_ranges(const MaskParams& m, int b, int p) {
  const int2* r = reinterpret_cast<const int2*>(m.ranges) + static_cast<size_t>(b) * m.max_ranges;
  int lo = INT_MAX, hi = INT_MIN;
  for (int i = 0; i < m.max_ranges; ++i) {
    const int2 e = __ldg(r + i);
    if (e.x < e.y && e.x <= p && p <= e.y) {
      lo = min(lo, e.x);
      hi = max(hi, e.y);
    }
  }
  return lo <= hi ? make_int2(lo, hi) : make_int2(-1, -1);
}

// The range entry of packed query row `row` (request b, position p): its
// table row, or in scan mode the scan of its request's ranges.
__device__ __forceinline__ int2 range_entry(const MaskParams& m, int row, int b, int p) {
  if (m.ranges != nullptr) return scan_ranges(m, b, p);
  if (!in_bounds(row, m.total_q, m.err)) return make_int2(-1, -1);
  return __ldg(reinterpret_cast<const int2*>(m.table) + row);
}

// p: absolute query position; k_len: keys of the request; use_range: the
// range part is on (row: packed row index, b: request, for range_entry).
__device__ __forceinline__ RowVis row_visibility(const MaskParams& m, int p, int k_len, bool use_range, int row,
                                                 int b) {
  const int2 e = use_range ? range_entry(m, row, b, p) : make_int2(1, 0);
  return row_visibility_from(m, p, k_len, use_range, e);
}

__device__ __forceinline__ RowVis row_visibility_from(const MaskParams& m, int p, int k_len, bool use_range, int2 e) {
  RowVis v;
  const long long wl = m.window_left, wr = m.window_right;
  long long lo = (wl >= 0) ? (long long)p - wl : 0;
  if (lo < 0) lo = 0;
  long long hi;
  if (m.causal) hi = p;
  else hi = (wr >= 0) ? (long long)p + wr : (long long)k_len - 1;
  if (hi > k_len - 1) hi = k_len - 1;
  v.b_lo = (int)lo;
  v.b_hi = (int)hi;
  v.r_lo = 1;
  v.r_hi = 0;
  if (use_range) {
    long long rl = e.x;
    if (wl >= 0 && (long long)p - wl > rl) rl = (long long)p - wl;
    if (rl < 0) rl = 0;
    long long rh = e.y;
    if (rh > k_len - 1) rh = k_len - 1;
    v.r_lo = (int)rl;
    v.r_hi = (int)rh;
  }
  return v;
}

// Row of a paged K/V cache (vLLM-style block table, block size
// 2^block_shift) that holds key l of request b: the block id of l's block
// times the block size plus l's offset in it.  Keys at or past the request's
// last block reuse its last block id (they are masked anyway), so the table
// is only read inside the request's blocks.
__device__ __forceinline__ int kv_row(const MaskParams& m, int b, int /*k0*/, int k_len, int l) {
  const int last = k_len > 0 ? ((k_len - 1) >> m.block_shift) : 0;
  const int blk = min(l >> m.block_shift, last);
  if (!in_bounds(blk, m.max_blocks, m.err)) return 0;
  const int id = __ldg(m.block_table + static_cast<size_t>(b) * m.max_blocks + blk);
  // unsigned: a corrupt id wraps instead of overflowing; TMA bounds-checks the row
  return static_cast<int>((static_cast<unsigned>(id) << m.block_shift) +
                          static_cast<unsigned>(l & ((1 << m.block_shift) - 1)));
}

// Whether the range part of the mask is on: scan mode, or a table whose
// covered flag (when given) is non-zero.
__device__ __forceinline__ bool table_active(const MaskParams& m) {
  if (m.ranges != nullptr) return true;
  if (m.table == nullptr) return false;
  if (m.covered == nullptr) return true;
  return *reinterpret_cast<const volatile int32_t*>(m.covered) != 0;
}

}  // namespace mvp
