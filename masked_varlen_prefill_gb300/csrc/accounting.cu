// Analytical work accounting of one attention call, on the host.
//
// Three levels, from coarse to exact to what the kernels execute:
//
//  1. The MFU/MBU estimate of vLLM PR #55624 ("Support Sliding Window
//     Attention and hybrid layers in MFU/MBU estimation"), ExecutionContext
//     with the window clamp: every request contributes num_tokens x
//     min(context_len, sliding_window) token-context products (the full
//     context without a window), attn_qk and attn_av each cost 2 x heads x
//     head_dim FLOPs per product, and a decode request reads
//     min(context_len, sliding_window) keys and values per KV head.  The
//     page's risk section calls this an upper bound that ignores the prefill
//     triangle and was never reconciled with profiler counts.
//  2. The exact visible (query row, key) pairs of the mask this library
//     computes: per row the union of the causal / window interval and the
//     window-clamped range interval.
//  3. The work this library's kernels execute for the call: the prefill
//     kernel's items and key tiles (the tile plan of attn_prefill.cu), the
//     tcgen05.mma instructions they issue and their FLOPs, the compulsory
//     bytes, and the keys the decode kernel reads (tiles aligned to its tile
//     size).  These are the figures a profiler's tensor-instruction and DRAM
//     counters measure.
//
// Declarations and contracts are in include/mvp.h.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <utility>
#include <vector>

#include "../../include/mvp.h"
#include "mvp_internal.cuh"

namespace mvp {
namespace {

struct Interval {
  long long lo, hi;  // closed; empty when lo > hi
  long long size() const { return hi >= lo ? hi - lo + 1 : 0; }
};

struct Row {
  Interval base, range;
  Interval hull() const {
    if (base.size() == 0) return range;
    if (range.size() == 0) return base;
    return {std::min(base.lo, range.lo), std::max(base.hi, range.hi)};
  }
  long long visible() const {
    const long long ov = std::max(0LL, std::min(base.hi, range.hi) - std::max(base.lo, range.lo) + 1);
    return base.size() + range.size() - (base.size() && range.size() ? ov : 0);
  }
};

// Visibility of the query at absolute position p (the interval rule of the
// attention contract: causal / window base OR the window-clamped range).
Row row_at(long long p, long long k_len, int causal, int wl, int wr, const int32_t* table_row) {
  Row r;
  r.base.lo = wl >= 0 ? std::max(0LL, p - wl) : 0;
  r.base.hi = causal ? p : (wr >= 0 ? p + wr : k_len - 1);
  r.base.hi = std::min(r.base.hi, k_len - 1);
  r.range = {1, 0};
  if (table_row != nullptr) {
    long long lo = table_row[0], hi = table_row[1];
    if (wl >= 0) lo = std::max(lo, p - wl);
    lo = std::max(lo, 0LL);
    hi = std::min(hi, k_len - 1);
    r.range = {lo, hi};
  }
  return r;
}

int pow2_divisor(int g, int cap) {
  int p = 1;
  while (p * 2 <= cap && g % (p * 2) == 0) p *= 2;
  return p;
}

}  // namespace
}  // namespace mvp

extern "C" int mvp_attn_accounting(const int32_t* cu_seqlens_q, const int32_t* seq_lens_k,
                                   const int32_t* context_lens, const int32_t* range_table, int num_reqs,
                                   int num_heads_q, int num_heads_kv, int head_dim, int causal, int window_left,
                                   int window_right, int variant, mvp_attn_counts* out) {
  using namespace mvp;
  if (out == nullptr) return MVP_ERR_ARG;
  *out = mvp_attn_counts{};
  if (num_reqs < 0 || num_heads_q < 1 || num_heads_kv < 1 || num_heads_q % num_heads_kv != 0) return MVP_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256 && head_dim != 512) return MVP_ERR_UNSUPPORTED;
  if ((causal != 0 && causal != 1) || window_left < -1 || window_right < -1) return MVP_ERR_ARG;
  if (variant != MVP_VARIANT_DEFAULT && variant != MVP_VARIANT_D512_HEAD_SPLIT) return MVP_ERR_ARG;
  if (variant == MVP_VARIANT_D512_HEAD_SPLIT && head_dim != 512) return MVP_ERR_UNSUPPORTED;
  if (num_reqs > 0 && (cu_seqlens_q == nullptr || seq_lens_k == nullptr)) return MVP_ERR_ARG;
  for (int b = 0; b < num_reqs; ++b) {
    const long long ql = static_cast<long long>(cu_seqlens_q[b + 1]) - cu_seqlens_q[b];
    const long long ctx = context_lens ? context_lens[b] : static_cast<long long>(seq_lens_k[b]) - ql;
    if (ql < 0 || seq_lens_k[b] < 0 || ctx < 0) return MVP_ERR_ARG;
  }
  if (num_reqs > 0 && cu_seqlens_q[0] != 0) return MVP_ERR_ARG;

  const double hq = num_heads_q, hkv = num_heads_kv, d = head_dim;
  const int group = num_heads_q / num_heads_kv;
  const PrefillShape shape = prefill_tile_shape(head_dim, variant == MVP_VARIANT_D512_HEAD_SPLIT);
  const int gpack = pow2_divisor(group, 8);
  const int n_hgroups = group / gpack;
  const long long item_pos = shape.item_rows / gpack;  // query positions of an item
  const long long bn = shape.bn;
  const int kt = decode_keys_per_tile(head_dim);
  const int per_cta = decode_heads_per_cta(head_dim, group);
  const int n_sub = (group + per_cta - 1) / per_cta;
  const long long sw = window_left >= 0 ? static_cast<long long>(window_left) + 1 : -1;  // tokens kept

  double tc = 0.0, dec_ctx = 0.0;
  long long vis_pre = 0, vis_dec = 0;
  long long items = 0, tiles = 0, touched_pre = 0, keys_walked = 0, rows_pre = 0, rows_dec = 0;
  for (int b = 0; b < num_reqs; ++b) {
    const long long q0 = cu_seqlens_q[b];
    const long long ql = cu_seqlens_q[b + 1] - q0;
    const long long kl = seq_lens_k[b];
    const long long ctx = context_lens ? context_lens[b] : kl - ql;
    if (ql == 0) continue;
    // 1. the page's estimate: num_tokens x min(context_len, window)
    const long long clamp = sw >= 0 ? std::min(kl, sw) : kl;
    tc += static_cast<double>(ql) * clamp;
    if (ql == 1) dec_ctx += clamp;
    // 2. exact visible pairs; 3. executed work
    const int32_t* tb = range_table ? range_table + 2 * q0 : nullptr;
    if (ql == 1) {
      const Row r = row_at(ctx, kl, causal, window_left, window_right, tb);
      vis_dec += r.visible();
      Interval h = r.hull();
      if (h.size() > 0) {
        h.lo &= ~static_cast<long long>(kt - 1);
        keys_walked += ((h.size() + kt - 1) / kt) * kt;
      }
      ++rows_dec;
      continue;
    }
    rows_pre += ql;
    std::vector<Interval> spans;
    for (long long pos0 = 0; pos0 < ql; pos0 += item_pos) {
      long long lo = LLONG_MAX, hi = LLONG_MIN;
      const long long pend = std::min(ql, pos0 + item_pos);
      for (long long i = pos0; i < pend; ++i) {
        const Row r = row_at(ctx + i, kl, causal, window_left, window_right, tb ? tb + 2 * i : nullptr);
        vis_pre += r.visible();
        const Interval h = r.hull();
        if (h.size() > 0) {
          lo = std::min(lo, h.lo);
          hi = std::max(hi, h.hi);
        }
      }
      if (lo > hi) continue;
      const long long kb_lo = lo / bn, n = hi / bn - kb_lo + 1;
      ++items;
      tiles += n;
      spans.push_back({kb_lo * bn, std::min((kb_lo + n) * bn, kl) - 1});
    }
    std::sort(spans.begin(), spans.end(), [](const Interval& a, const Interval& c) { return a.lo < c.lo; });
    long long cur_lo = 0, cur_hi = -1;
    for (const Interval& s : spans) {
      if (s.lo > cur_hi + 1) {
        touched_pre += cur_hi - cur_lo + 1;
        cur_lo = s.lo;
        cur_hi = s.hi;
      } else {
        cur_hi = std::max(cur_hi, s.hi);
      }
    }
    touched_pre += cur_hi - cur_lo + 1;
  }

  const double heads_items = hkv * n_hgroups * shape.dv_split;  // items per (request, q tile)
  out->est_token_context_product = tc;
  out->est_attn_qk_flops = 2.0 * hq * d * tc;
  out->est_attn_av_flops = 2.0 * hq * d * tc;
  out->est_decode_kv_read_bytes = 2.0 * hkv * d * 2.0 * dec_ctx;
  out->visible_prefill = vis_pre;
  out->visible_decode = vis_dec;
  out->exact_flops = 4.0 * d * hq * static_cast<double>(vis_pre + vis_dec);
  out->exact_decode_kv_bytes = 2.0 * hkv * d * 2.0 * static_cast<double>(vis_dec);
  out->prefill_items = static_cast<long long>(items * heads_items);
  out->prefill_tiles = static_cast<long long>(tiles * heads_items);
  // per tile, each issuing CTA: qk_k / 16 QK MMAs (M x BN x 16) and BN / 16
  // PV MMAs (M x (oc + rowsum_n) x 16: where the tensor core sums the rows,
  // the PV MMA carries rowsum_n more columns)
  out->prefill_mma_instructions = out->prefill_tiles * shape.issuers * (shape.qk_k / 16 + shape.bn / 16);
  out->prefill_mma_flops = static_cast<double>(out->prefill_tiles) * shape.issuers * 2.0 * shape.mma_m *
                           static_cast<double>(bn) * (shape.qk_k + shape.oc + shape.rowsum_n);
  out->prefill_compulsory_bytes = 2.0 * static_cast<double>(rows_pre) * hq * d * 2.0 +  // q in, out
                                  2.0 * static_cast<double>(touched_pre) * hkv * d * 2.0;  // k, v
  out->decode_keys_walked = keys_walked;
  out->decode_read_bytes = static_cast<double>(keys_walked) * hkv * d * 2.0 * 2.0 +
                           static_cast<double>(rows_dec) * hq * d * 2.0;
  out->decode_cta_read_bytes = static_cast<double>(keys_walked) * hkv * n_sub * d * 2.0 * 2.0 +
                               static_cast<double>(rows_dec) * hq * d * 2.0;
  return MVP_OK;
}
