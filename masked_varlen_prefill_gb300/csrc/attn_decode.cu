// Masked varlen attention forward, single-token (decode) rows, sm_103a.
//
// The step14_4 "Causal Mask optimisation" tutorial observes that a decode
// query (seq_len == 1) needs no mask construction: it sees a contiguous run
// of keys.  Here such a row's visible keys are the interval
// [max(0, p - window_left), p] (plus, in general, the range part of
// mask.cuh), read once per KV head for all the query heads that share it.
//
// This path is HBM-bound (each key is 2 * D bf16 of K and V used by G query
// heads), so it is SIMT, not tensor-core work:
// * A CTA handles one (request, KV head, key split).  A producer warp streams
//   KT-key tiles of K and V into a 2- or 3-stage shared-memory ring with TMA;
//   four compute warps read them back conflict-free.
// * A warp takes a step of KG keys at a time.  Scores: the DS lanes that
//   share one key each form partial dot products over their slice of the
//   head dimension for every q head of the CTA, and a shuffle reduce-scatter
//   over those DS lanes leaves each lane the full score of one (key, head)
//   pair.  The online base-2 softmax (lazy rescale) follows, and the p * V
//   accumulation with lane l owning D/32 dimensions of every head.
// * Long rows are split across CTAs (split-KV); partial (acc, max, sum)
//   triples are merged by decode_combine_kernel.  Without workspace every row
//   is a single split and the CTA writes the final output itself.
#include <cuda_bf16.h>

#include <mutex>

#include "mask.cuh"
#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {

namespace {

constexpr int kMaxStages = 3;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

__host__ __device__ constexpr int kt_for(int d) { return d == 64 ? 128 : (d == 128 ? 64 : 32); }
// Stages of the K/V ring.  D = 128: two, so that three CTAs (12 compute warps)
// fit an SM's shared memory; with three stages (two CTAs per SM) the decode
// rows of the mixed serving batches ran at 87 / 82 % of the measured HBM
// bandwidth against 98 / 90 % with two.  The other head dims keep three: their
// CTAs are limited by registers, so fewer stages would only shrink the bytes
// in flight.
__host__ __device__ constexpr int stages_for(int d) { return d == 128 ? 2 : 3; }
__host__ __device__ constexpr int box_for(int d) { return d > 256 ? 256 : d; }
// Compute warps per CTA (a producer warp comes on top).  Eight at D = 128
// (two CTAs per SM, 8-dim lane slices to fit the registers) measured slower
// than four with three CTAs per SM.
__host__ __device__ constexpr int nw_for(int) { return 4; }
// Dims of q and K per lane in the score step (q registers: QDL * GP): 16
// keeps the reduce-scatter to log2(D / 16) stages; 8-dim slices at D = 128
// and 4 heads (one more stage, fewer registers) measured ~10 % slower.
__host__ __device__ constexpr int qdl_for(int, int gp) { return gp == 8 ? 8 : 16; }
// (key, head) probabilities each lane owns per warp step.  Two at D = 128
// with four or more heads per CTA: 16-key steps give every warp two
// independent score chains and halve the per-step softmax overhead; on a
// part of the SMs (beside the prefill kernel) the decode rows of the mixed
// serving batch ran 11 % faster.  A 64-key tile then holds exactly one step
// per compute warp.
__host__ __device__ constexpr int pairs_for(int d, int gp) { return (d == 128 && gp >= 4) ? 2 : 1; }

template <int D>
struct DCfg {
  static constexpr int DPL = D / 32;          // dims per lane
  static constexpr int KT = kt_for(D);        // keys per tile
  static constexpr int BOX = box_for(D);
  static constexpr int NBOX = D / BOX;
  static constexpr int TILE = KT * D * 2;     // bytes of one K (or V) tile
  static constexpr int STAGES = stages_for(D);
  static constexpr int SMEM = STAGES * 2 * TILE + 1024;
  static constexpr int NW = nw_for(D);          // compute warps
  static constexpr int THREADS = (NW + 1) * 32;  // + the producer warp
};

struct __align__(8) DBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  WaitCtl wc;  // abort flag and wait budget of this CTA
};

template <int DPL>
__device__ __forceinline__ void load_row(const uint8_t* p, float (&x)[DPL]) {
  if constexpr (DPL == 2) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    x[0] = __uint_as_float(u << 16);
    x[1] = __uint_as_float(u & 0xffff0000u);
  } else if constexpr (DPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
#pragma unroll
    for (int c = 0; c < DPL / 8; ++c) {
      const uint4 u = *reinterpret_cast<const uint4*>(p + c * 16);
      x[8 * c + 0] = __uint_as_float(u.x << 16); x[8 * c + 1] = __uint_as_float(u.x & 0xffff0000u);
      x[8 * c + 2] = __uint_as_float(u.y << 16); x[8 * c + 3] = __uint_as_float(u.y & 0xffff0000u);
      x[8 * c + 4] = __uint_as_float(u.z << 16); x[8 * c + 5] = __uint_as_float(u.z & 0xffff0000u);
      x[8 * c + 6] = __uint_as_float(u.w << 16); x[8 * c + 7] = __uint_as_float(u.w & 0xffff0000u);
    }
  }
}

// Byte offset of (key kk, this lane's dims) inside a tile stored as NBOX
// boxes of [KT][BOX] bf16.
template <int D>
__device__ __forceinline__ int row_off(int kk, int lane) {
  using C = DCfg<D>;
  const int dim0 = lane * C::DPL;
  const int box = dim0 / C::BOX;
  return box * (C::KT * C::BOX * 2) + kk * (C::BOX * 2) + (dim0 % C::BOX) * 2;
}

// PAGED: K/V rows come through a block table (compile-time, so the packed
// kernel carries none of the paged addressing).
template <int D, int GP, bool PAGED>
__global__ void __launch_bounds__(DCfg<D>::THREADS)
    attn_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                       const DecodeParams p) {
  using C = DCfg<D>;
  constexpr int DPL = C::DPL;
  constexpr int PPL = pairs_for(D, GP);  // probabilities per lane and step
  constexpr int KG = 32 * PPL / GP;      // keys per warp step
  constexpr int NG = C::KT / KG;     // warp steps per tile
  static_assert(C::NW * GP * (D + 2) * 4 <= C::STAGES * 2 * C::TILE, "merge buffers fit the stages");
  static_assert(C::KT % KG == 0, "whole steps per tile");
  extern __shared__ uint8_t smem_raw[];
  // Per compute warp, the step's 32 probabilities (key kk, head g at
  // kk * GP + g) as (p, p) pairs, read back by every lane as broadcasts
  // instead of 32 shuffles.
  __shared__ __align__(16) float pbuf[C::NW][64 * pairs_for(D, GP)];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DBarriers sb;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sp = blockIdx.x;
  const int b = blockIdx.y;
  const int n_sub = (p.group + GP - 1) / GP;
  const int hkv = blockIdx.z / n_sub;
  const int sub = blockIdx.z % n_sub;
  const int hq0 = hkv * p.group + sub * GP;       // first q head of this CTA
  const int heads_here = min(GP, p.group - sub * GP);

  const int q0 = __ldg(p.m.cu_q + b);
  const int q_len = __ldg(p.m.cu_q + b + 1) - q0;
  if (q_len != 1) return;
  if (!in_bounds(q0, p.total_q, p.err)) return;  // (bounds-checked build; the whole CTA)
  int k0, k_len;
  if constexpr (PAGED) {
    k0 = 0;
    k_len = __ldg(p.m.seq_k + b);
  } else {
    k0 = __ldg(p.m.cu_k + b);
    k_len = __ldg(p.m.cu_k + b + 1) - k0;
  }
  (void)in_bounds(0, k_len, p.err);  // a decode row needs a key: q_len <= k_len (checked build)
  const int pos = p.m.ctx_lens ? __ldg(p.m.ctx_lens + b) : (k_len - 1);
  const RowVis vis = row_visibility(p.m, pos, k_len, table_active(p.m), q0, b);
  int lo, hi;
  vis.hull(lo, hi);
  // Tiles start on multiples of KT (the keys before the visible set are
  // masked): a tile never straddles a cache block of a paged layout (block
  // sizes and KT are powers of two), and packed and paged calls walk the
  // same tiles.
  if (lo <= hi) lo &= ~(C::KT - 1);
  const int c_lo = lo + sp * p.chunk;
  const int c_hi = (lo <= hi) ? min(hi, c_lo + p.chunk - 1) : -1;
  const int n_keys = (lo <= hi && c_lo <= c_hi) ? (c_hi - c_lo + 1) : 0;
  const int n_tiles = (n_keys + C::KT - 1) / C::KT;
  const bool single = p.partial == nullptr;
  if (n_keys == 0 && !single) {
    // An empty split still publishes a neutral partial for the combine.
    float* part = p.partial + ((static_cast<size_t>(b) * p.hq + hq0) * p.n_splits + sp) * (D + 2);
    for (int g = 0; g < heads_here; ++g) {
      float* pg = part + static_cast<size_t>(g) * p.n_splits * (D + 2);
      for (int d = threadIdx.x; d < D + 2; d += blockDim.x) pg[d] = (d == D) ? -INFINITY : 0.f;
    }
    return;
  }
  if (n_keys == 0 && sp > 0) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sb.full[s], 1);
      mbar_init(&sb.empty[s], C::NW);
    }
    sb.wc.abort = 0;
    sb.wc.limit_us = p.m.wait_limit_us;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == C::NW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      const int kbox = PAGED ? min(C::KT, 1 << p.m.block_shift) : C::KT;
      int issued = 0;
      bool ok = true;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % C::STAGES;
        if (t >= C::STAGES &&
            !mbar_wait(&sb.empty[s], ((t / C::STAGES) - 1) & 1, &sb.wc, p.err, kDevTimeoutLoad)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sb.full[s], 2 * C::TILE);
        uint8_t* ks = smem + s * 2 * C::TILE;
        uint8_t* vs = ks + C::TILE;
        // one box per run of keys inside one cache block (the whole tile when packed)
        for (int r = 0; r < C::KT; r += kbox) {
          const int row = PAGED ? kv_row(p.m, b, k0, k_len, c_lo + t * C::KT + r) : k0 + c_lo + t * C::KT + r;
#pragma unroll
          for (int x = 0; x < C::NBOX; ++x) {
            tma_load_3d(ks + x * (C::KT * C::BOX * 2) + r * (C::BOX * 2), &map_k, &sb.full[s], x * C::BOX, hkv, row);
            tma_load_3d(vs + x * (C::KT * C::BOX * 2) + r * (C::BOX * 2), &map_v, &sb.full[s], x * C::BOX, hkv, row);
          }
        }
        ++issued;
      }
      if (!ok) sb.wc.abort = 1;
      WaitCtl own_flag = own_wait_ctl(&sb.wc);
      for (int s = 0; s < C::STAGES && s < issued; ++s) {
        const int last = ((issued - 1 - s) / C::STAGES) * C::STAGES + s;
        mbar_wait(&sb.full[s], (last / C::STAGES) & 1, &own_flag, nullptr, 0);
      }
    }
    return;
  }

  // ------------------------------------------------------------------ compute
  // Scores: DS lanes share one key's dot product, each over QDL dims (two or
  // one 16-byte chunks of the K row: chunk ds + j * DS, so that with DS >= 8
  // the eight lanes of a quarter-warp read 128 consecutive bytes), for all GP
  // heads at once; a
  // reduce-scatter over those DS lanes leaves each lane the full score of one
  // (key, head) pair, held by DUP lanes alike.  A warp step of KG keys runs
  // NSUB such sub-steps of KS keys, so that every lane owns the probabilities
  // of PPL of the step's 32 * PPL (key, head) pairs.
  constexpr int QDL = qdl_for(D, GP);     // dims per lane in the score step
  constexpr int DS = D / QDL;              // lanes per key
  constexpr int KS = 32 / DS;              // keys per sub-step
  constexpr int DUP = DS / GP;             // lanes holding the same score
  constexpr int NSUB = DUP * PPL;          // sub-steps per warp step
  constexpr int QCH = QDL / 8;             // 16-byte chunks of a K row per lane
  static_assert(DS >= GP && DS <= 32 && KS * NSUB == KG, "score layout");
  const int ds = lane % DS;   // dim slice
  const int ks = lane / DS;   // key of the sub-step
  const int hh = ds / DUP;    // head of this lane's scores
  const int rr = ds % DUP;    // this lane keeps the scores of sub-steps rr + r * DUP, r < PPL

  // q for this lane's dim chunks, every head of the CTA, pre-scaled to log2
  // units, as (even, odd) dim pairs for the packed fp32x2 FMAs.
  uint64_t q2[GP][QDL / 2];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
#pragma unroll
    for (int j = 0; j < QCH; ++j) {
      float tmp[8];
#pragma unroll
      for (int d = 0; d < 8; ++d) tmp[d] = 0.f;
      if (g < heads_here) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) +
                             ((static_cast<size_t>(q0) * p.hq + hq0 + g) * D + 8 * (ds + j * DS)) * 2;
        load_row<8>(src, tmp);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        q2[g][4 * j + i] = f2_pack(tmp[2 * i] * p.m.scale_log2, tmp[2 * i + 1] * p.m.scale_log2);
    }
  }
  const bool key0_mode = p.m.sink_mode == 1 && p.m.sinks != nullptr;
  float my_sink = 0.f;
  if (key0_mode && hh < heads_here) my_sink = __ldg(p.m.sinks + hq0 + hh) * 1.4426950408889634f;
  // Keys every lane may take without a mask test: inside the split and in
  // the interval the row sees whole (key 0 excluded when it carries a sink).
  int core_lo, core_hi;
  vis.core(core_lo, core_hi);
  core_hi = min(core_hi, c_hi);
  if (key0_mode) core_lo = max(core_lo, 1);

  // Per-step probabilities as (p, p) pairs, [key of the step][head], read
  // back by every lane as broadcasts.
  uint64_t* pb = reinterpret_cast<uint64_t*>(pbuf[warp]);

  // O partial sums: lane l owns dims [l * DPL, (l + 1) * DPL) of every head.
  constexpr int DP2 = DPL / 2;
  uint64_t acc2[GP][DP2];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int i = 0; i < DP2; ++i) acc2[g][i] = 0ull;  // (+0.f, +0.f)
  // Running max of head hh in log2 units, raised only when a step's max
  // exceeds it by more than kRescaleThreshold (probabilities stay <= 2^8),
  // and this lane's share of that head's sum.
  float m_h = -INFINITY;
  float l_part = 0.f;

  bool ok = true;
  for (int t = 0; t < n_tiles && ok; ++t) {
    const int s = t % C::STAGES;
    if (!mbar_wait(&sb.full[s], (t / C::STAGES) & 1, &sb.wc, p.err, kDevTimeoutLoad)) {
      ok = false;
      break;
    }
    const uint8_t* ks_tile = smem + s * 2 * C::TILE;
    const uint8_t* vs_tile = ks_tile + C::TILE;
    const int t0 = c_lo + t * C::KT;
    const bool interior = t0 >= core_lo && t0 + C::KT - 1 <= core_hi;
    for (int gi = warp; gi < NG; gi += C::NW) {
      float x[NSUB];
#pragma unroll
      for (int a = 0; a < NSUB; ++a) {
        const int kk = gi * KG + a * KS + ks;  // key of the tile
        uint64_t a2[GP];
#pragma unroll
        for (int j = 0; j < QCH; ++j) {
          const int dim0 = 8 * (ds + j * DS);
          float kr[8];
          load_row<8>(ks_tile + (dim0 / C::BOX) * (C::KT * C::BOX * 2) + kk * (C::BOX * 2) + (dim0 % C::BOX) * 2,
                      kr);
          uint64_t k2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) k2[i] = f2_pack(kr[2 * i], kr[2 * i + 1]);
#pragma unroll
          for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              a2[g] = (j == 0 && i == 0) ? f2_mul(q2[g][0], k2[0]) : f2_fma(q2[g][4 * j + i], k2[i], a2[g]);
        }
        float v[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          float ae, ao;
          f2_unpack(a2[g], ae, ao);
          v[g] = ae + ao;
        }
        // reduce-scatter over the DS lanes of the key: while more than one
        // head is left, the upper lanes keep the upper half; then plain sums
#pragma unroll
        for (int o = DS / 2, n = GP / 2; o >= 1; o >>= 1, n >>= 1) {
          if (n >= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n; ++i) {
              const float send = upper ? v[i] : v[i + n];
              const float keep = upper ? v[i + n] : v[i];
              v[i] = keep + __shfl_xor_sync(kFull, send, o);
            }
          } else {
            v[0] += __shfl_xor_sync(kFull, v[0], o);
          }
        }
        x[a] = v[0];
        if (!interior) {
          const int key = t0 + kk;
          if (key0_mode && key == 0) x[a] += my_sink;
          if (!(key <= c_hi && vis.visible(key))) x[a] = -INFINITY;
        }
      }
      // max of head hh over the step's keys: this lane's NSUB, then the KS keys
      float mx = x[0];
#pragma unroll
      for (int a = 1; a < NSUB; ++a) mx = fmaxf(mx, x[a]);
#pragma unroll
      for (int o = DS; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const bool need = mx > m_h + kRescaleThreshold;
      if (__any_sync(kFull, need)) {
        const float alpha = need ? ex2_approx(m_h - mx) : 1.f;  // 0 while m_h is -inf
        if (need) m_h = mx;
        l_part *= alpha;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float ag = __shfl_sync(kFull, alpha, g * DUP);
          const uint64_t a2 = f2_pack(ag, ag);
#pragma unroll
          for (int i = 0; i < DP2; ++i) acc2[g][i] = f2_mul(acc2[g][i], a2);
        }
      }
#pragma unroll
      for (int r = 0; r < PPL; ++r) {  // this lane's pairs: sub-steps rr + r * DUP
        float xr = x[r * DUP];
#pragma unroll
        for (int a = 1; a < DUP; ++a) xr = (rr == a) ? x[r * DUP + a] : xr;
        const float pr = (xr == -INFINITY) ? 0.f : ex2_approx(xr - m_h);
        l_part += pr;
        pb[((r * DUP + rr) * KS + ks) * GP + hh] = f2_pack(pr, pr);
      }
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < KG; ++kk) {
        float vr[DPL];
        load_row<DPL>(vs_tile + row_off<D>(gi * KG + kk, lane), vr);
        uint64_t v2[DP2];
#pragma unroll
        for (int i = 0; i < DP2; ++i) v2[i] = f2_pack(vr[2 * i], vr[2 * i + 1]);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const uint64_t pg2 = pb[kk * GP + g];  // same address in every lane: broadcast
#pragma unroll
          for (int i = 0; i < DP2; ++i) acc2[g][i] = f2_fma(pg2, v2[i], acc2[g][i]);
        }
      }
      __syncwarp();  // every lane has read pbuf before the next step writes it
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sb.empty[s]);
  }

  // per-head sums: the lanes holding head hh (every key, every duplicate)
#pragma unroll
  for (int o = 1; o < DUP; o <<= 1) l_part += __shfl_xor_sync(kFull, l_part, o);
#pragma unroll
  for (int o = DS; o < 32; o <<= 1) l_part += __shfl_xor_sync(kFull, l_part, o);

  // ------------------------------------------------------------------ merge warps
  // Stage buffers are free once every tile was consumed by every warp.
  asm volatile("bar.sync 1, %0;" ::"r"(C::NW * 32) : "memory");
  float* sm = reinterpret_cast<float*>(smem);                 // [NW][GP][D]
  float* sml = sm + C::NW * GP * D;                            // [NW][GP][2]
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int i = 0; i < DP2; ++i) {
      float x0, x1;
      f2_unpack(acc2[g][i], x0, x1);
      sm[(warp * GP + g) * D + lane * DPL + 2 * i] = x0;
      sm[(warp * GP + g) * D + lane * DPL + 2 * i + 1] = x1;
    }
  if (ks == 0 && rr == 0) {  // lane hh * DUP: head hh's max and sum
    sml[(warp * GP + hh) * 2 + 0] = m_h;
    sml[(warp * GP + hh) * 2 + 1] = l_part;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(C::NW * 32) : "memory");

  const bool null_mode = p.m.sink_mode == 2 && p.m.sinks != nullptr;
  for (int idx = threadIdx.x; idx < heads_here * D; idx += C::NW * 32) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, sml[(w * GP + g) * 2]);
    float a = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
      const float mw = sml[(w * GP + g) * 2];
      const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      a += f * sm[(w * GP + g) * D + d];
      L += f * sml[(w * GP + g) * 2 + 1];
    }
    const int h = hq0 + g;
    if (!single) {
      float* part = p.partial + ((static_cast<size_t>(b) * p.hq + h) * p.n_splits + sp) * (D + 2);
      part[d] = a;
      if (d == 0) {
        part[D] = M;
        part[D + 1] = L;
      }
    } else {
      if (null_mode) {
        const float sk = __ldg(p.m.sinks + h) * 1.4426950408889634f;
        const float M2 = fmaxf(M, sk);
        const float f = (M == -INFINITY) ? 0.f : ex2_approx(M - M2);
        a *= f;
        L = L * f + ex2_approx(sk - M2);
        M = M2;
      }
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      reinterpret_cast<__nv_bfloat16*>(p.out)[(static_cast<size_t>(q0) * p.hq + h) * D + d] =
          __float2bfloat16_rn(a * inv);
      if (d == 0 && p.lse != nullptr) {
        const float mu = (M == -INFINITY) ? 0.f : M;
        p.lse[static_cast<size_t>(h) * p.total_q + q0] =
            (L > 0.f) ? (mu + lg2_approx(L)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }
  (void)ok;
}

// One warp per (request, q head): merge the split partials of a decode row.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
  const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.num_reqs * p.hq) return;
  const int b = warp_global / p.hq;
  const int h = warp_global % p.hq;
  const int q0 = __ldg(p.m.cu_q + b);
  if (__ldg(p.m.cu_q + b + 1) - q0 != 1) return;
  if (!in_bounds(q0, p.total_q, p.err)) return;  // (bounds-checked build)
  const float* part = p.partial + (static_cast<size_t>(b) * p.hq + h) * p.n_splits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, part[s * (D + 2) + D]);
  const bool null_mode = p.m.sink_mode == 2 && p.m.sinks != nullptr;
  float sk = 0.f;
  if (null_mode) {
    sk = __ldg(p.m.sinks + h) * 1.4426950408889634f;
    M = fmaxf(M, sk);
  }
  float L = null_mode ? ex2_approx(sk - M) : 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const float ms = part[s * (D + 2) + D];
    if (ms != -INFINITY) L += part[s * (D + 2) + D + 1] * ex2_approx(ms - M);
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  for (int d = lane; d < D; d += 32) {
    float a = 0.f;
    for (int s = 0; s < p.n_splits; ++s) {
      const float ms = part[s * (D + 2) + D];
      if (ms != -INFINITY) a += part[s * (D + 2) + d] * ex2_approx(ms - M);
    }
    reinterpret_cast<__nv_bfloat16*>(p.out)[(static_cast<size_t>(q0) * p.hq + h) * D + d] =
        __float2bfloat16_rn(a * inv);
  }
  if (lane == 0 && p.lse != nullptr) {
    const float mu = (M == -INFINITY) ? 0.f : M;
    p.lse[static_cast<size_t>(h) * p.total_q + q0] =
        (L > 0.f) ? (mu + lg2_approx(L)) * 0.6931471805599453f : -INFINITY;
  }
}

// The dynamic shared memory attribute of each instantiation is set once per
// device (under a mutex: two host threads may make their first call on a
// device at the same time).
std::mutex g_decode_attr_mutex;

template <int D, int GP>
cudaError_t launch_dg(const DecodeParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream) {
  const bool paged = p.m.block_table != nullptr;
  auto kern = paged ? attn_decode_kernel<D, GP, true> : attn_decode_kernel<D, GP, false>;
  static bool attr_set[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(g_decode_attr_mutex);
    if (!attr_set[paged ? 1 : 0][dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<D>::SMEM);
      if (e != cudaSuccess) return e;
      attr_set[paged ? 1 : 0][dev] = true;
    }
  }
  const int n_sub = (p.group + GP - 1) / GP;
  dim3 grid(p.n_splits, p.num_reqs, p.hkv * n_sub);
  kern<<<grid, DCfg<D>::THREADS, DCfg<D>::SMEM, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream,
                     int* launches) {
  // Heads per CTA: the group padded to a power of two, capped so that q and
  // the accumulators (2 * GP * D / 32 floats per lane) stay in registers.
  cudaError_t e;
  if (p.group == 1) e = launch_dg<D, 1>(p, mk, mv, stream);
  else if (p.group == 2) e = launch_dg<D, 2>(p, mk, mv, stream);
  else if (p.group <= 4 || D >= 512) e = launch_dg<D, 4>(p, mk, mv, stream);
  else if constexpr (D < 512) e = launch_dg<D, 8>(p, mk, mv, stream);
  else e = cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  ++*launches;
  if (p.partial != nullptr) {
    const int warps = p.num_reqs * p.hq;
    decode_combine_kernel<D><<<(warps + 3) / 4, 128, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  return cudaSuccess;
}

}  // namespace

int decode_keys_per_tile(int head_dim) { return kt_for(head_dim); }
int decode_box_inner(int head_dim) { return box_for(head_dim); }

cudaError_t launch_decode(int head_dim, const DecodeParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                          cudaStream_t stream, int* launches) {
  switch (head_dim) {
    case 64: return launch_d<64>(p, mk, mv, stream, launches);
    case 128: return launch_d<128>(p, mk, mv, stream, launches);
    case 256: return launch_d<256>(p, mk, mv, stream, launches);
    case 512: return launch_d<512>(p, mk, mv, stream, launches);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mvp
