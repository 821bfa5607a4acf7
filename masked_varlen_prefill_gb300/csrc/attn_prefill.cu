// Masked varlen attention forward, prefill rows: tcgen05 + TMA, sm_103a.
//
// Computes, for 128-row query tiles, softmax(scale * Q K^T + mask) V with the
// online (running max / running sum) formulation in base 2, as the Triton
// kernel of vLLM PR #49815 does ("Key source snippets", the sinks branch of
// _fwd_kernel: exp2 domain, sink * log2(e), null-logit init m = sink, l = 1, or
// key-0 bias added to the masked score of key 0).  The mask is the
// (causal AND window) OR range rule of vLLM PR #50294's mask_mod, evaluated as
// two closed key intervals per row (mask.cuh).
//
// GB300 design (not the pages' kernels):
// * Work item = NCTA 128-row tiles.  With GQA, G_pack query heads of one KV
//   head share a tile: row r is (position r / G_pack, head h0 + r % G_pack), so
//   a K/V tile read from L2 serves G_pack heads.  The Q tile is a single 3-D
//   TMA box (64 dims, G_pack heads, 128 / G_pack positions), 128-byte swizzled.
// * D = 128, 256 and 512 run as CTA pairs (a 2-CTA cluster, tcgen05
//   .cta_group::2): each MMA is M = 256 (each CTA's 128 rows, scores and O in
//   its own TMEM), each CTA loads only half of every K tile (its keys) and half
//   of every V tile (its value columns), and rank 0 issues the MMAs for both.
//   A tile costs each SM half the L2 -> shared-memory bytes and half the
//   shared memory, which buys two K and two V stages at D = 256 and 512.
// * Persistent CTAs (one per SM) take the items, numbered q tile fastest so
//   that concurrent CTAs share K/V windows in L2, with a static stride; the
//   last round comes from a work queue in the caller's workspace, so the tail
//   goes to whichever CTA frees up first.  A scheduler warp computes each item's
//   geometry and key-tile plan (a warp reduction over the item's rows) into a
//   ring that every role reads, and
//   all barrier phases run on CTA-wide counters, so the producer and the MMA
//   issuer move on to the next item's Q, K and QK while the softmax warps
//   still finish the current item.
// * Warp roles: warp 0 issues TMA loads, warp 1 allocates TMEM and issues
//   tcgen05.mma from one thread, and SPLIT softmax warpgroups (warps 2..)
//   own the rows: with BN = 128 two warpgroups split every row's 128 scores
//   into halves of 64 (warps w and w+4 read the same TMEM lanes), exchange the
//   row max through shared memory once per tile, and split the O correction
//   and epilogue by columns.
// * TMEM (512 columns): S double buffer [0, BN) and [BN, 2 BN) in fp32; the
//   bf16 probabilities P overwrite the first BN/2 columns of their S buffer and
//   feed O += P V as the TMEM operand of tcgen05.mma; O at [2 BN, 2 BN + DV).
//   At D = 128 the PV MMA also multiplies P by a block of ones that follows
//   each V stage in shared memory, so that the row sums of P (what O is
//   normalised by) accumulate in TMEM beside O instead of costing the softmax
//   warps an unpack and an add per score pair.
// * MMA order per step j: S_j = Q K_j^T, then O += P_{j-1} V_{j-1}, so the
//   tensor core computes the next scores while the softmax warps work on the
//   current ones.  MMA descriptors are computed once; loads are released per
//   tile (each extra tcgen05.commit or wait costs the single issuing thread).
// * Key tiles are visited only inside [min hull, max hull] of the tile's rows;
//   tiles fully inside every row's all-visible interval skip the mask.
// * O is rescaled lazily: a row's reference max only moves when the new max
//   exceeds it by more than 2^8 (probabilities then stay <= 256).
// * Every mbarrier wait is bounded (ptx.cuh).
#include <cuda_bf16.h>

#include <mutex>

#include "mask.cuh"
#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {

namespace {

constexpr int kBM = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr unsigned kFullMask = 0xffffffffu;

template <int D_, int DV_, int BN_, int KST_, int VST_, int NCTA_, int SPLITD_ = 0, int NS_ = 2, int ROWSUM_ = 0>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int DV = DV_;        // value columns handled by one item
  static constexpr int BN = BN_;        // keys per tile
  static constexpr int KST = KST_;      // K tile stages
  static constexpr int VST = VST_;      // V tile stages
  static constexpr int NCTA = NCTA_;    // CTAs of a cluster working on one item (1 or 2)
  // Two ways for two CTAs to share an item: a pair (M split: each CTA owns
  // 128 of the 256 rows, rank 0 issues .cta_group::2 MMAs) or a head-dim
  // split (SPLITD: both CTAs own the same 128 rows; each multiplies its half
  // of the head dimension into a partial score and its half of the value
  // columns into its own O, issuing its own MMAs; the partial scores are
  // summed through distributed shared memory).
  static constexpr bool SPLITD = SPLITD_ != 0;
  static constexpr bool PAIR = NCTA == 2 && !SPLITD;
  static constexpr int MMA_CTAS = PAIR ? 2 : 1;  // CTAs one MMA spans
  static constexpr int DQ = SPLITD ? D / 2 : D;  // head dims of Q and K held by one CTA
  static constexpr int KROWS = BN / MMA_CTAS;    // keys of a K tile loaded by one CTA
  static constexpr int DVC = DV / NCTA;          // value columns of a V tile loaded by one CTA
  static constexpr int OC = SPLITD ? DVC : DV;   // O columns in this CTA's TMEM
  static constexpr int ITEM_ROWS = kBM * MMA_CTAS;
  static constexpr int QCH = DQ / 64;   // 64-dim chunks of Q and K (one TMA box each)
  static constexpr int VCH = DVC / 64;  // 64-column chunks of this CTA's part of a V tile
  static constexpr int DV_SPLIT = D / DV;
  static constexpr int SPLIT = BN / 64;         // softmax warpgroups (column halves of a row)
  static constexpr int HC = BN / SPLIT;         // score columns per softmax thread (64)
  static constexpr int HDV = OC / SPLIT;        // O columns per softmax thread (rescale)
  // Warp layout: warpgroup 0 = TMA producer (warp 0), MMA issuer (1), plan
  // scheduler (2), one idle warp; SPLIT softmax warpgroups; one epilogue
  // warpgroup that reads O out of TMEM and stores the output rows.
  static constexpr int PRODUCER_WARP = 0;
  static constexpr int MMA_WARP = 1;
  static constexpr int SCHED_WARP = 2;
  static constexpr int SOFTMAX_BEGIN = 4;
  static constexpr int SOFTMAX_END = SOFTMAX_BEGIN + 4 * SPLIT;
  static constexpr int EPI_BEGIN = SOFTMAX_END;
  static constexpr int WARPS = EPI_BEGIN + 4;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int CONSUMER_WARPS = 2 + 4 * SPLIT + 4;  // warps that read the plan ring
  // Register split for 512 threads (128 each at launch): the softmax warps
  // get 168, warpgroup 0 and the epilogue 88 each (sum 4 x 128).
  static constexpr bool REG_SPLIT = SPLIT == 2;
  static constexpr int REGS_CTRL = 88;
  static constexpr int REGS_SOFTMAX = 168;
  static constexpr int REGS_EPI = 88;
  static_assert(!REG_SPLIT || (THREADS == 512 && REGS_CTRL + 2 * REGS_SOFTMAX + REGS_EPI <= 4 * 128),
                "register split");
  static constexpr int Q_BYTES = kBM * DQ * 2;
  static constexpr int K_BYTES = KROWS * DQ * 2;  // per CTA
  static constexpr int V_BYTES = BN * DVC * 2;    // per CTA, loaded per tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_BYTES;
  static constexpr int V_OFF = K_OFF + KST * K_BYTES;
  // Row sums by the tensor core (ROWSUM): each V stage is followed by a
  // constant 64-column block of bf16 ones, and the PV MMA takes ONES more
  // columns of B from each CTA (its value columns, then ONES of the ones), so
  // that the accumulator holds, after each CTA's part of O, ONES copies of
  // every row's sum of the bf16 probabilities, accumulated and rescaled with
  // O.  The softmax warps then add only the unrounded probabilities (for the
  // LSE).  A V stage is VCH blocks of BN x 128 bytes (the loaded value
  // columns) plus the ones block.
  static constexpr bool ROWSUM = ROWSUM_ != 0;
  // Otherwise the softmax warps sum the rounded probabilities by
  // mixed-precision adds (add.rn.f32.bf16 on each bf16 half, no unpack; the
  // same bits as unpacking and adding): measured 58.5 vs 57.6 % of the bf16
  // peak at D = 512 and 0.3 % faster at D = 256 than a shift / mask / packed
  // add (once the MMA warp issued fewer instructions; before, the latter
  // was 0.5-1 % faster there).
  static constexpr bool MIXED_SUM = !ROWSUM;
  static constexpr int ONES = ROWSUM ? 16 : 0;
  static constexpr int V_STAGE = (VCH + (ROWSUM ? 1 : 0)) * BN * 128;  // stage stride
  static constexpr int PART = DVC + ONES;                           // accumulator columns per CTA part
  static constexpr int OCW = SPLITD ? OC : MMA_CTAS * PART;         // accumulator columns (PV N)
  static constexpr int TILE_BYTES = V_OFF + VST * V_STAGE;
  // SPLITD: the peer's partial scores of two tiles, [2][128 rows][BN] fp32
  static constexpr int XS_OFF = TILE_BYTES;
  static constexpr int XS_BYTES = SPLITD ? 2 * kBM * BN * 4 : 0;
  static constexpr int RED_OFF = XS_OFF + XS_BYTES;  // column-half exchange slots: [2 parity][SPLIT][128] float2
  static constexpr int RED_BYTES = SPLIT > 1 ? 2 * SPLIT * kBM * 8 : 0;
  // Hand-off slots softmax -> epilogue: (1 / l, LSE) per row and item.  Two
  // when they fit (the D = 512 tiles leave room for one).
  static constexpr int ROW_OFF = RED_OFF + RED_BYTES;
  static constexpr int EPI_SLOTS = (ROW_OFF + 2 * kBM * 8 + 1024 + 1024 <= 227 * 1024) ? 2 : 1;
  // Paged K/V: the producer warp caches the block ids of its current and next
  // item here (two buffers of IDS_CAP ids): up to 2048 each, what fits (none
  // at D = 512).
  static constexpr int IDS_OFF = ROW_OFF + EPI_SLOTS * kBM * 8;
  static constexpr int ids_cap(int cap) {
    return cap < 64 ? 0 : (IDS_OFF + 2 * cap * 4 + 1024 + 1024 <= 227 * 1024 ? cap : ids_cap(cap / 2));
  }
  static constexpr int IDS_CAP = ids_cap(2048);
  static constexpr int SMEM_BYTES = IDS_OFF + 2 * IDS_CAP * 4 + 1024;  // + alignment slack
  // S buffers in TMEM.  The MMA issuer runs QK NS - 1 tiles ahead of PV:
  // with two, S_{j+2} can only be computed once P_j (every softmax warp's)
  // has been handed over and PV_j issued; with three, S_{j+2} is computed
  // while the softmax warps still work on tile j.  (Three fit next to O at
  // D = 128 only, which gives those columns to the row sums instead: with
  // the softmax warps' row-sum work gone, two buffers measured as fast as
  // three.)
  static constexpr int NS = NS_;
  // S buffer of CTA-wide tile t (t >= 0) and the phase of its barriers; the
  // unsigned forms keep NS = 2 at a mask and a shift.
  static __device__ __forceinline__ uint32_t sbuf(int t) { return static_cast<uint32_t>(t) % NS; }
  static __device__ __forceinline__ uint32_t sphase(int t) { return (static_cast<uint32_t>(t) / NS) & 1u; }
  static constexpr int S_COL = 0;
  static constexpr int O_COL = NS * BN;
  static constexpr int L_COL = O_COL + DVC;  // ROWSUM: the row sum (first ones column of part 0)
  static constexpr int TMEM_COLS = 512;
  static_assert(O_COL + OCW <= TMEM_COLS, "TMEM budget");
  // (each softmax half's O columns lie in one part; the ones block sits on a
  // 64-column boundary of the stage, LBO = BN x 128 bytes away)
  static_assert(!ROWSUM || (PAIR && HDV == DVC && DVC % 64 == 0 && OCW <= 256), "row sums in the PV MMA");
  // Accumulator column of the item's value column `d` (0 .. OC - 1).
  static __host__ __device__ constexpr int ocol(int d) { return (d / DVC) * PART + d % DVC; }
  static_assert(NS == 2 || NS == 3, "S buffers");
  static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
  static_assert(BN == 64 || BN == 128, "BN");
  static_assert(DV % 64 == 0 && OC <= 256 && DVC % 64 == 0, "DV");
  static_assert(NCTA == 1 || NCTA == 2, "NCTA");
  static_assert(!SPLITD || (NCTA == 2 && SPLIT == 1 && DV == D), "head-dim split: one softmax warpgroup, no DV split");
  static_assert(HDV % 32 == 0, "O columns per thread");
  static_assert(KST >= 1 && KST <= 4 && VST >= 1 && VST <= 4, "stages");
  // With two K and two V stages, "K stage of tile t free" is exactly "S_t
  // computed" (s_full[t & 1]) and "V stage of tile t free" is "O += P_t V_t
  // done" (o_done[t & 1]); the Q buffer is free once the item's last S is.
  // The single MMA-issuing thread then commits twice per tile instead of
  // four or five times (its issue rate bounds the tensor pipe).
  static constexpr bool MERGED_RELEASE = KST == 2 && VST == 2;
  static_assert(!MERGED_RELEASE || NS == 2, "merged release reads stage frees off the two S buffers");
  static_assert(!SPLITD || NS == 2, "head-dim split: two S buffers");
};

// One work item: NCTA 128-row query tiles of one request and one KV head
// group ((for D = 512) one half of the value dimension), with its key-tile
// plan.  pos0 is the item's first query position; CTA rank r of a pair owns
// positions pos0 + r * 128 / G_pack onwards.
struct Item {
  int b, pos0, q0, q_len, k0, k_len, ctx, h0, hkv, dv0;
  bool valid;
};

struct Plan {
  int kb_lo, n_tiles, int_lo, int_hi;
};

struct PlanEntry {
  Item it;
  Plan pl;
  int last;  // 1: no more items for this CTA
};

constexpr int kPlanRing = 4;
// Work queue: items claimed ahead of the producer's loads.  The softmax warps
// take the next item's plan as they start an item (to load its rows' inputs
// early), so one claim ahead leaves them waiting on the claim and plan at
// every item start; two hide that behind a whole item.
constexpr int kClaimAhead = 2;
// Rounds of items (one per CTA or pair) at the end of the item space that
// come from the work queue; the rounds before keep the static stride.
constexpr int kQueueRounds = 1;

struct __align__(8) Barriers {
  uint64_t plan_full[kPlanRing];
  uint64_t plan_empty[kPlanRing];
  PlanEntry plans[kPlanRing];
  uint64_t claim_full[kPlanRing];   // work queue, pair: rank 0 wrote the item it claimed into claims[i] of rank 1
  uint64_t claim_empty[kPlanRing];  // ... and rank 1 has read it (rank 0's barrier)
  int claims[kPlanRing];
  uint64_t plan_taken[kPlanRing];  // work queue: the producer took the entry in slot i
  int n_static;                    // scheduler: items walked with the static stride
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[4];
  uint64_t v_empty[4];
  uint64_t s_full[3];  // tile t: buffer t % NS
  uint64_t p_full[3];
  uint64_t o_done[2];
  uint64_t final_mma;
  uint64_t epi_full[2];   // an item's (1 / l, LSE) rows are written (half-0 softmax warps)
  uint64_t epi_empty[2];  // ... and read (epilogue warps)
  uint64_t o_free;        // O of the previous item is out of TMEM (rank 0; arrivals from both CTAs)
  uint64_t x_full[2];     // head-dim split: the peer's partial scores of a tile are in slot i
  uint64_t x_empty[2];    // ... the peer has read what this CTA sent into its slot i
  uint64_t xchg[4][2];  // softmax column-half pairs (per TMEM lane quarter), by parity
  uint32_t tmem_base;
  WaitCtl wc;  // abort flag and wait budget of this CTA
};

// Items are numbered q tile fastest (latest tile first), then head group,
// then request: the CTAs running at the same time then work on neighbouring
// tiles of a few (request, KV head) pairs, whose K/V windows overlap and stay
// in L2, and every CTA's strided sequence mixes heavy and light tiles.
template <class C, bool PAGED>
__device__ __forceinline__ Item item_geometry(int item, const PrefillParams& p) {
  const int nz = p.hkv * p.n_hgroups * C::DV_SPLIT;
  const int x = item % p.n_qtiles;  // 0 = latest q tile (heaviest under causal masks)
  const int rest = item / p.n_qtiles;
  const int z = rest % nz;
  Item it;
  it.b = rest / nz + p.req_offset;
  it.dv0 = (z % C::DV_SPLIT) * C::DV;
  const int hz = z / C::DV_SPLIT;
  it.hkv = hz / p.n_hgroups;
  it.h0 = it.hkv * (p.hq / p.hkv) + (hz % p.n_hgroups) * p.gpack;
  it.q0 = __ldg(p.m.cu_q + it.b);
  it.q_len = __ldg(p.m.cu_q + it.b + 1) - it.q0;
  if constexpr (PAGED) {
    it.k0 = 0;
    it.k_len = __ldg(p.m.seq_k + it.b);
  } else {
    it.k0 = __ldg(p.m.cu_k + it.b);
    it.k_len = __ldg(p.m.cu_k + it.b + 1) - it.k0;
  }
  it.ctx = p.m.ctx_lens ? __ldg(p.m.ctx_lens + it.b) : (it.k_len - it.q_len);
  if (it.q_len > 0) (void)in_bounds(it.q_len - 1, it.k_len, p.err);  // q_len <= k_len (checked build)
  it.pos0 = (p.n_qtiles - 1 - x) * (C::ITEM_ROWS / p.gpack);
  it.valid = it.pos0 < it.q_len && !(p.skip_decode && it.q_len == 1);
  return it;
}

// The first item after an invalid item `item` (geometry `it`) that can have
// rows: the first item of this (request, head) block whose q tile has rows,
// or, when the request has no prefill rows at all, the first item of the
// next request that has (32 requests tested per step by the warp); the
// scheduler then takes the first item of its own sequence at or after it.
// Item spaces sized for a capacity (upper-bound q lengths, padding requests)
// then cost O(requests) per CTA, not O(items).  Warp-collective; LLONG_MAX
// past the last request.
template <class C>
__device__ __forceinline__ long long candidate_target(int item, const Item& it, const PrefillParams& p, int lane) {
  const int nz = p.hkv * p.n_hgroups * C::DV_SPLIT;
  const long long per_req = static_cast<long long>(nz) * p.n_qtiles;
  const int prows = C::ITEM_ROWS / p.gpack;  // query positions per item
  long long target;
  if (it.q_len > 0 && !(p.skip_decode && it.q_len == 1)) {
    const int x_min = p.n_qtiles - (it.q_len + prows - 1) / prows;  // first x with pos0 < q_len
    target = static_cast<long long>(item / p.n_qtiles) * p.n_qtiles + x_min;
    if (target <= item) target = item + 1;  // (rows past max_q_len: not computed)
  } else {
    int b = it.b + 1;
    for (;;) {
      if (b >= p.num_reqs) return LLONG_MAX;
      const int c = b + lane;
      bool good = false;
      if (c < p.num_reqs) {
        const int ql = __ldg(p.m.cu_q + c + 1) - __ldg(p.m.cu_q + c);
        good = ql > 0 && !(p.skip_decode && ql == 1);
      }
      const unsigned m = __ballot_sync(kFullMask, good);
      if (m != 0u) {
        b += __ffs(m) - 1;
        break;
      }
      b += 32;
    }
    target = (b - p.req_offset) * per_req;
  }
  return target;
}

// Work-queue words (the prefill scheduler's, in the caller's workspace):
// (launch tag << 32) | counter, the tag being this launch's %gridid.
// queue_add adds 1 to the counter and returns its old value, or -1 when the
// word keeps changing hands (another launch uses it at the same time; a
// device error is recorded).  check: first use in this launch; a word that
// carries another tag gets this one with the counter at 1 (returns 0).
__device__ __forceinline__ long long queue_add(unsigned long long* word, bool check, int* err) {
  const unsigned long long tag = grid_launch_id() << 32;
  if (check) {
    for (int tries = 0;; ++tries) {
      const unsigned long long cur = atomicAdd(word, 0ull);
      if ((cur & 0xffffffff00000000ull) == tag) break;
      if (atomicCAS(word, cur, tag | 1ull) == cur) return 0;
      if (tries > (1 << 16)) {
        atomicCAS(err, 0, kDevQueueConflict);
        return -1;
      }
    }
  }
  const unsigned long long v = atomicAdd(word, 1ull);
  if ((v & 0xffffffff00000000ull) != tag) {
    atomicCAS(err, 0, kDevQueueConflict);
    return -1;
  }
  return static_cast<long long>(v & 0xffffffffull);
}

// A claiming CTA is done (also after an abort): count it in the second
// word; the launch's last one resets both counters under its tag, so that a
// later launch carrying the same tag (a graph replay) starts at item 0.  The
// fences order every CTA's claims before its count, and the last count before
// the reset.
__device__ __forceinline__ void queue_finish(unsigned long long* words, int n_claimers, int* err) {
  __threadfence();
  if (queue_add(words + 1, true, err) == n_claimers - 1) {
    __threadfence();
    const unsigned long long tag = grid_launch_id() << 32;
    atomicExch(words, tag);
    atomicExch(words + 1, tag);
  }
}

// Key-tile plan of an item (warp-collective, over all NCTA * 128 rows, so
// both CTAs of a pair walk the same tiles): the tiles between the smallest
// and largest visible key of any row, and the tiles inside every row's
// all-visible interval (no mask needed there).
template <class C>
__device__ __forceinline__ Plan plan_tiles(const Item& it, const PrefillParams& p, bool use_table, int lane) {
  int hl_min = INT_MAX, hh_max = INT_MIN, cl_max = INT_MIN, ch_min = INT_MAX;
#pragma unroll
  for (int k = 0; k < C::ITEM_ROWS / 32; ++k) {
    const int row = lane + 32 * k;
    const int qi = it.pos0 + row / p.gpack;
    if (qi < it.q_len) {
      const RowVis v = row_visibility(p.m, it.ctx + qi, it.k_len, use_table, it.q0 + qi, it.b);
      int hl, hh, cl, ch;
      v.hull(hl, hh);
      v.core(cl, ch);
      if (hl <= hh) {
        hl_min = min(hl_min, hl);
        hh_max = max(hh_max, hh);
      }
      cl_max = max(cl_max, cl);  // an empty core (INT_MAX, INT_MIN) removes the interior
      ch_min = min(ch_min, ch);
    }
  }
  hl_min = __reduce_min_sync(kFullMask, hl_min);
  hh_max = __reduce_max_sync(kFullMask, hh_max);
  cl_max = __reduce_max_sync(kFullMask, cl_max);
  ch_min = __reduce_min_sync(kFullMask, ch_min);
  Plan pl{0, 0, 1, 0};
  if (hl_min <= hh_max) {
    pl.kb_lo = hl_min / C::BN;
    pl.n_tiles = hh_max / C::BN - pl.kb_lo + 1;
    if (cl_max <= ch_min) {
      pl.int_lo = (cl_max + C::BN - 1) / C::BN;
      pl.int_hi = (ch_min + 1) / C::BN - 1;
    }
  }
  return pl;
}

// Warp-collective: take plan entry n from the ring (written by the scheduler
// warp) and release its slot.
__device__ __forceinline__ bool consume_plan(Barriers& sb, int n, int lane, PlanEntry& e, int* err) {
  const int slot = n % kPlanRing;
  const bool ok = mbar_wait(&sb.plan_full[slot], (n / kPlanRing) & 1, &sb.wc, err, kDevTimeoutOther);
  e = sb.plans[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(&sb.plan_empty[slot]);
  return ok;
}

// The two column halves of a row (warps w and w+4) swap one float2 through
// shared memory.  Exchange k uses slot and barrier k & 1 (the partner cannot
// overwrite slot k & 1 before this thread has passed exchange k + 1).  The
// wait is bounded, so a failed partner cannot hang the pair.
__device__ __forceinline__ bool pair_exchange(float2* slots, uint64_t* xb, int& k, int half, int row, float2 mine,
                                              float2& theirs, volatile WaitCtl* abort_flag, int* err) {
  float2* slot = slots + (k & 1) * (2 * kBM);
  slot[half * kBM + row] = mine;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&xb[k & 1]);  // release: the warp's slots are visible
  const bool ok = mbar_wait(&xb[k & 1], (k >> 1) & 1, abort_flag, err, kDevTimeoutSoftmax);
  theirs = slot[(1 - half) * kBM + row];
  ++k;
  return ok;
}

__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* r) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// In a pair, TMA copies of both CTAs complete on rank 0's barrier.
template <class C>
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, uint64_t* full, int x, int y, int z) {
  if constexpr (C::PAIR) tma_load_3d_pair(dst, map, mapa_shared(smem_u32(full), 0), x, y, z);
  else tma_load_3d(dst, map, full, x, y, z);
}

// PAGED: K/V rows come through a block table (compile-time, so the packed
// kernel carries none of the paged addressing).  LSE: the caller asked for
// the log-sum-exp, so the softmax warps also sum the unrounded
// probabilities; without it they skip that packed add per score pair (O
// does not depend on it).
template <class C, bool PAGED, bool LSE>
__global__ void __launch_bounds__(C::THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Barriers sb;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = p.n_qtiles * (p.num_reqs - p.req_offset) * p.hkv * p.n_hgroups * C::DV_SPLIT;
  constexpr int BN = C::BN;
  const int rank = C::NCTA == 2 ? static_cast<int>(cluster_rank()) : 0;
  const bool leader = !C::PAIR || rank == 0;  // issues its MMAs and owns the "full" barriers
  // This CTA's first query position within an item (a pair's rank 1 owns the
  // second 128 rows) and first head dim of Q and K (a head-dim split's rank 1
  // owns the second half); evaluated inside each role, so that no register
  // stays live across the roles' register split.
  auto row_pos_off = [&]() { return C::PAIR ? rank * (kBM / p.gpack) : 0; };
  auto dq_off = [&]() { return C::SPLITD ? rank * C::DQ : 0; };

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPlanRing; ++i) {
      mbar_init(&sb.plan_full[i], 1);
      mbar_init(&sb.plan_empty[i], C::CONSUMER_WARPS - (leader ? 0 : 1));  // a pair's rank 1 issues no MMAs
    }
    for (int i = 0; i < kPlanRing; ++i) {
      mbar_init(&sb.claim_full[i], 1);
      mbar_init(&sb.claim_empty[i], 1);
    }
    mbar_init(&sb.q_full, 1);
    mbar_init(&sb.q_empty, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
    }
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 4 * C::SPLIT * C::MMA_CTAS);  // one arrival per softmax warp
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sb.o_done[i], 1);
    mbar_init(&sb.final_mma, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.epi_full[i], 4);
      mbar_init(&sb.epi_empty[i], 4);
    }
    mbar_init(&sb.o_free, 4 * C::MMA_CTAS);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.x_full[i], 4);   // head-dim split: the peer's four softmax warps wrote their partial scores
      mbar_init(&sb.x_empty[i], 4);  // ... and read this CTA's
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&sb.xchg[i][0], 2);
      mbar_init(&sb.xchg[i][1], 2);
    }
    sb.wc.abort = 0;
    sb.wc.limit_us = p.m.wait_limit_us;
    for (int i = 0; i < kPlanRing; ++i) mbar_init(&sb.plan_taken[i], 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    if constexpr (C::PAIR) {
      tmem_alloc_pair(&sb.tmem_base, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&sb.tmem_base, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  if constexpr (C::ROWSUM) {
    // the ones block after each V stage (bf16 1.0), made visible to the tensor core
    constexpr int kWords = C::BN * 128 / 16;  // 16-byte words per block
#pragma unroll 1
    for (int i = threadIdx.x; i < C::VST * kWords; i += C::THREADS)
      reinterpret_cast<uint4*>(smem + C::V_OFF + (i / kWords) * C::V_STAGE + C::VCH * C::BN * 128)[i % kWords] =
          make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (C::NCTA == 2) cluster_sync_all();  // the peer's barriers are initialised
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;
  // Launched with programmatic serialization: the setup above overlapped the
  // previous kernel in the stream (the range fill); every global input,
  // including the table's covered flag, is read after this point.
  griddep_wait();
  const bool use_table = table_active(p.m);

  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;


  if (warp < C::SOFTMAX_BEGIN) {
    if constexpr (C::REG_SPLIT) regs_decrease<C::REGS_CTRL>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // Loads follow the order in which the MMA issuer frees the buffers: per
      // item Q and K_0, then per step j K_{j+1} and V_j.  The next item's Q and
      // K_0 go out before the current item's last V tile: they wait only for
      // the last QK, which the tensor core finishes before the PV that frees
      // that V stage.  Stage counters run across items.
      if (lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
      }
      bool ok = true;
      int n = 0, qn = 0, kc = 0, vc = 0;  // plans taken, Q / K / V tiles issued
      // Next item that has key tiles (warp-collective); false at the end.
      auto next_item = [&](PlanEntry& e) -> bool {
        for (;;) {
          if (!consume_plan(sb, n++, lane, e, p.err)) {
            ok = false;
            return false;
          }
          if (lane == 0 && p.queue != nullptr) mbar_arrive(&sb.plan_taken[(n - 1) % kPlanRing]);
          if (e.last) return false;
          if (e.pl.n_tiles > 0) return true;
        }
      };
      const int pos_off = row_pos_off();
      const int dq0 = dq_off();
      // L2 warming: an item's Q tile and first K / V tiles come from DRAM,
      // with a latency several times a tile's MMA time, while its later tiles
      // follow at the pace of the pipeline.  The next item's Q and (packed
      // K / V) first kPrefetchAhead K / V tiles are prefetched while the
      // current item runs; each CTA of a pair warms its own half.  Prefetching
      // further tiles inside an item measured slower (extra TMA requests),
      // and so did K / V prefetch for paged caches at every block size.
      constexpr int kPrefetchAhead = 2;
      // Paged K/V: loads go one block run at a time (box heights capped at the
      // block size on the host).
      const int kbox = PAGED ? min(C::KROWS, 1 << p.m.block_shift) : C::KROWS;
      const int vbox = PAGED ? min(BN, 1 << p.m.block_shift) : BN;
      // Block ids of an item's key range, copied into shared memory by the
      // whole warp (cp.async) while the item before it runs, so that the
      // issuing lane never waits on a block-table load; buffer `buf` (items
      // alternate) holds the ids of the blocks from the item's first one on.
      int32_t* ids = reinterpret_cast<int32_t*>(smem + C::IDS_OFF);
      int ids_plan = -1;  // plan whose ids are in flight into the other buffer
      auto cache_ids = [&](const PlanEntry& e, int buf, bool wait) {
        if constexpr (PAGED && C::IDS_CAP > 0) {
          const int sh = p.m.block_shift;
          const int fb = (e.pl.kb_lo * BN) >> sh;
          const int last = e.it.k_len > 0 ? (e.it.k_len - 1) >> sh : 0;
          const int nb = min((((e.pl.kb_lo + e.pl.n_tiles) * BN - 1) >> sh) - fb + 1, C::IDS_CAP);
          const int32_t* row = p.m.block_table + static_cast<size_t>(e.it.b) * p.m.max_blocks;
          for (int i = lane; i < nb; i += 32) {
            const int blk = min(fb + i, last);
            if (in_bounds(blk, p.m.max_blocks, p.err)) cp_async_4(ids + buf * C::IDS_CAP + i, row + blk);
          }
          cp_async_commit();
          if (wait) {
            cp_async_wait_all();
            __syncwarp();
          }
        }
      };
      // Cache row of key `key` of item e (packed: the packed row).
      auto row_of = [&](const PlanEntry& e, int buf, int key) -> int {
        if constexpr (PAGED) {
          if constexpr (C::IDS_CAP > 0) {
            const int sh = p.m.block_shift;
            const int last = e.it.k_len > 0 ? (e.it.k_len - 1) >> sh : 0;
            const int idx = min(key >> sh, last) - ((e.pl.kb_lo * BN) >> sh);
            if (static_cast<unsigned>(idx) < static_cast<unsigned>(C::IDS_CAP))
              return static_cast<int>((static_cast<unsigned>(ids[buf * C::IDS_CAP + idx]) << sh) +
                                      static_cast<unsigned>(key & ((1 << sh) - 1)));
          }
          return kv_row(p.m, e.it.b, e.it.k0, e.it.k_len, key);
        } else {
          return e.it.k0 + key;
        }
      };
      int cbuf = 0;  // ids buffer of the current item
      auto prefetch_kv = [&](const PlanEntry& e, int j) {  // packed K / V only
        const int key0 = e.it.k0 + (e.pl.kb_lo + j) * BN;
#pragma unroll
        for (int c = 0; c < C::QCH; ++c)
          tma_prefetch_l2_3d(&map_k, dq0 + c * 64, e.it.hkv, key0 + (C::PAIR ? rank * C::KROWS : 0));
#pragma unroll
        for (int c = 0; c < C::VCH; ++c)
          tma_prefetch_l2_3d(&map_v, e.it.dv0 + rank * C::DVC + c * 64, e.it.hkv, key0);
      };
      // Plan n (the next one to consume) if the scheduler has published it;
      // never waits (warp-collective: every lane observes the plan itself).
      // The slot cannot be reused before this warp consumes it.  Paged: the
      // plan's block ids start on their way into the other ids buffer, whose
      // item issued its last load before the warp's last sync.
      // Returns false while plan n is not published yet (then retried; the
      // test is non-blocking, so the loads it sits between are not delayed).
      auto prefetch_next_item = [&]() -> bool {
        const int slot = n % kPlanRing;
        if (!__all_sync(kFullMask, mbar_test_wait(&sb.plan_full[slot], (n / kPlanRing) & 1))) return false;
        const PlanEntry e = sb.plans[slot];
        if (e.last || e.pl.n_tiles == 0) return true;
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < C::QCH; ++c)
            tma_prefetch_l2_3d(&map_q, dq0 + c * 64, e.it.h0, e.it.q0 + e.it.pos0 + pos_off);
          for (int j = 0; !PAGED && j < kPrefetchAhead && j < e.pl.n_tiles; ++j) prefetch_kv(e, j);
        }
        if constexpr (PAGED) {
          cache_ids(e, cbuf ^ 1, false);
          ids_plan = n;
        }
        return true;
      };
      auto load_q = [&](const PlanEntry& e) -> bool {
        if (qn > 0) {
          bool free;
          if constexpr (C::MERGED_RELEASE) {
            const int tl = kc - 1;  // the previous item's last tile
            free = mbar_wait(&sb.s_full[tl & 1], (tl >> 1) & 1, &sb.wc, p.err, kDevTimeoutMma);
          } else {
            free = mbar_wait(&sb.q_empty, (qn - 1) & 1, &sb.wc, p.err, kDevTimeoutMma);
          }
          if (!free) return false;
        }
        if (leader) mbar_arrive_expect_tx(&sb.q_full, C::MMA_CTAS * C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::QCH; ++c)
          tma_load<C>(sQ + c * (kBM * 128), &map_q, &sb.q_full, dq0 + c * 64, e.it.h0, e.it.q0 + e.it.pos0 + pos_off);
        ++qn;
        return true;
      };
      auto load_k = [&](const PlanEntry& e, int j, int buf) -> bool {
        const int s = kc % C::KST;
        if (kc >= C::KST) {
          const int tp = kc - C::KST;  // the tile that used this stage before
          const bool free = C::MERGED_RELEASE
                                ? mbar_wait(&sb.s_full[tp & 1], (tp >> 1) & 1, &sb.wc, p.err, kDevTimeoutLoad)
                                : mbar_wait(&sb.k_empty[s], (tp / C::KST) & 1, &sb.wc, p.err, kDevTimeoutLoad);
          if (!free) return false;
        }
        if (leader) mbar_arrive_expect_tx(&sb.k_full[s], C::MMA_CTAS * C::K_BYTES);
        const int key0 = (e.pl.kb_lo + j) * BN + (C::PAIR ? rank * C::KROWS : 0);  // this CTA's first key of the tile
        if constexpr (PAGED) {
          // one box per run of K rows inside one cache block (a rolled loop:
          // the producer's code stays small next to the other roles')
#pragma unroll 1
          for (int r = 0; r < C::KROWS; r += kbox) {
            const int krow = row_of(e, buf, key0 + r);
#pragma unroll
            for (int c = 0; c < C::QCH; ++c)
              tma_load<C>(sK + s * C::K_BYTES + c * (C::KROWS * 128) + r * 128, &map_k, &sb.k_full[s],
                          dq0 + c * 64, e.it.hkv, krow);
          }
        } else {
#pragma unroll
          for (int c = 0; c < C::QCH; ++c)
            tma_load<C>(sK + s * C::K_BYTES + c * (C::KROWS * 128), &map_k, &sb.k_full[s], dq0 + c * 64, e.it.hkv,
                        e.it.k0 + key0);
        }
        ++kc;
        return true;
      };
      auto load_v = [&](const PlanEntry& e, int j, int buf) -> bool {
        const int s = vc % C::VST;
        if (vc >= C::VST) {
          const int tp = vc - C::VST;
          const bool free = C::MERGED_RELEASE
                                ? mbar_wait(&sb.o_done[tp & 1], (tp >> 1) & 1, &sb.wc, p.err, kDevTimeoutLoad)
                                : mbar_wait(&sb.v_empty[s], (tp / C::VST) & 1, &sb.wc, p.err, kDevTimeoutLoad);
          if (!free) return false;
        }
        if (leader) mbar_arrive_expect_tx(&sb.v_full[s], C::MMA_CTAS * C::V_BYTES);
        const int key0 = (e.pl.kb_lo + j) * BN;
        if constexpr (PAGED) {
#pragma unroll 1
          for (int r = 0; r < BN; r += vbox) {
            const int vrow = row_of(e, buf, key0 + r);
#pragma unroll
            for (int c = 0; c < C::VCH; ++c)
              tma_load<C>(sV + s * C::V_STAGE + c * (BN * 128) + r * 128, &map_v, &sb.v_full[s],
                          e.it.dv0 + rank * C::DVC + c * 64, e.it.hkv, vrow);
          }
        } else {
#pragma unroll
          for (int c = 0; c < C::VCH; ++c)
            tma_load<C>(sV + s * C::V_STAGE + c * (BN * 128), &map_v, &sb.v_full[s], e.it.dv0 + rank * C::DVC + c * 64,
                        e.it.hkv, e.it.k0 + key0);
        }
        ++vc;
        return true;
      };
      PlanEntry cur;
      bool have = next_item(cur);
      if (have) cache_ids(cur, cbuf, true);
      if (have && lane == 0) ok = load_q(cur) && load_k(cur, 0, cbuf);
      ok = __shfl_sync(kFullMask, ok, 0);
      while (ok && have) {
        const int nt = cur.pl.n_tiles;
        // (the next plan may be published while this item's tiles are issued)
        bool prefetched = false;
        for (int j = 0;; ++j) {
          if (!prefetched) prefetched = prefetch_next_item();
          if (!ok || j + 1 >= nt) break;
          if (lane == 0) {
            ok = load_k(cur, j + 1, cbuf);
            if (ok) ok = load_v(cur, j, cbuf);
          }
          ok = __shfl_sync(kFullMask, ok, 0);
        }
        PlanEntry nxt;
        const bool have_next = ok && next_item(nxt);
        if (PAGED && have_next) {
          if (ids_plan == n - 1) {  // prefetched while the current item ran
            cp_async_wait_all();
            __syncwarp();
          } else {
            cache_ids(nxt, cbuf ^ 1, true);
          }
        }
        ids_plan = -1;
        if (lane == 0 && ok) {
          if (have_next) ok = load_q(nxt) && load_k(nxt, 0, cbuf ^ 1);
          if (ok) ok = load_v(cur, nt - 1, cbuf);
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        cur = nxt;
        have = have_next;
        cbuf ^= 1;
      }
      if constexpr (PAGED) cp_async_wait_all();  // block ids still in flight
      // Drain: never leave the CTA with a TMA write still in flight.  Each
      // full barrier's last armed phase is waited for, ignoring the CTA abort
      // flag (issued copies always complete, and must before the CTA exits).
      // A pair's full barriers live in rank 0 and count both CTAs' copies;
      // rank 1 stays until rank 0 has drained (the final cluster barrier).
      if (lane == 0 && !leader && !ok) sb.wc.abort = 1;
      if (lane == 0 && leader) {
        if (!ok) sb.wc.abort = 1;
        WaitCtl own_flag = own_wait_ctl(&sb.wc);
        if (qn > 0) mbar_wait(&sb.q_full, (qn - 1) & 1, &own_flag, nullptr, 0);
        for (int i = 0; i < 4; ++i) {
          // stage i was last armed by tile i + KST * m, m = (issued - 1 - i) / KST (phase parity m)
          if (i < C::KST && kc > i) mbar_wait(&sb.k_full[i], ((kc - 1 - i) / C::KST) & 1, &own_flag, nullptr, 0);
          if (i < C::VST && vc > i) mbar_wait(&sb.v_full[i], ((vc - 1 - i) / C::VST) & 1, &own_flag, nullptr, 0);
        }
      }
    } else if (warp == 1 && leader) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop (converged, warp-uniform values); each
      // tcgen05.mma and commit is issued by one elected lane.  Descriptors are
      // computed once and each MMA only adds a compile-time offset.  Tile t is
      // the CTA-wide tile index: S buffer t % NS, K stage t % KST, V stage
      // t % VST.  In a pair, the same descriptors and TMEM addresses name the
      // operands in both CTAs.
      constexpr uint32_t idesc_qk = idesc_bf16_f32(C::ITEM_ROWS, C::BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(C::ITEM_ROWS, C::OCW, false, true);
      const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), BN * 128, 1024);
      const bool issuer = elect_one();  // issues the MMAs; the commits' elect.sync picks the same lane
      bool ok = true;
      int T = 0, qn = 0;
      for (int n = 0; ok; ++n) {
        PlanEntry e;
        ok = consume_plan(sb, n, lane, e, p.err);
        if (!ok || e.last) break;
        const Plan& pl = e.pl;
        if (pl.n_tiles == 0) continue;
        ok = mbar_wait_spin(&sb.q_full, qn & 1, &sb.wc, p.err, kDevTimeoutLoad);
        ++qn;
        // Step j issues S_j = Q K_j^T, then O += P V of tile j - LEAD.
        constexpr int LEAD = C::NS - 1;
        for (int j = 0; ok && j < pl.n_tiles + LEAD; ++j) {
          if (j < pl.n_tiles) {
            const int t = T + j;
            const int s = t % C::KST;
            if (!mbar_wait_spin(&sb.k_full[s], (t / C::KST) & 1, &sb.wc, p.err, kDevTimeoutLoad)) {
              ok = false;
              break;
            }
            const uint32_t d = tmem + C::S_COL + C::sbuf(t) * BN;
            const uint64_t dk = desc_add(dk0, static_cast<uint32_t>((s * C::K_BYTES) >> 4));
            if (issuer) {
#pragma unroll
              for (int c = 0; c < C::QCH; ++c) {
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16) {
                  const uint64_t a = desc_add(dq, static_cast<uint32_t>((c * (kBM * 128) + k16 * 32) >> 4));
                  const uint64_t b = desc_add(dk, static_cast<uint32_t>((c * (C::KROWS * 128) + k16 * 32) >> 4));
                  mma_ss_one<C::MMA_CTAS>(d, a, b, idesc_qk, (c | k16) != 0 ? 1u : 0u);
                }
              }
            }
            __syncwarp();
            if constexpr (!C::MERGED_RELEASE) {
              mma_commit_elect<C::MMA_CTAS>(&sb.k_empty[s]);
              if (j == pl.n_tiles - 1) mma_commit_elect<C::MMA_CTAS>(&sb.q_empty);  // Q free for the next item
            }
            mma_commit_elect<C::MMA_CTAS>(&sb.s_full[C::sbuf(t)]);
          }
          if (j >= LEAD) {
            const int t = T + j - LEAD;
            // (a suspending wait: this warp shares its SM sub-partition with
            // the softmax warps of TMEM lane quarter 1, and polling for the
            // softmax's hand-off took their issue slots, so that in a
            // per-warp trace those warps arrived last on most tiles)
            if (!mbar_wait(&sb.p_full[C::sbuf(t)], C::sphase(t), &sb.wc, p.err, kDevTimeoutSoftmax)) {
              ok = false;
              break;
            }
            // The item's first PV overwrites O: the epilogue warps must have
            // read the previous item's O out of TMEM (both CTAs of a pair).
            if (j == LEAD && qn > 1 &&
                !mbar_wait_spin(&sb.o_free, (qn - 2) & 1, &sb.wc, p.err, kDevTimeoutSoftmax)) {
              ok = false;
              break;
            }
            const int s = t % C::VST;
            if (!mbar_wait_spin(&sb.v_full[s], (t / C::VST) & 1, &sb.wc, p.err, kDevTimeoutLoad)) {
              ok = false;
              break;
            }
            tc_fence_after();  // P (softmax warps) and the O read-out (epilogue warps) are ordered before
            const uint32_t pcol = tmem + C::S_COL + C::sbuf(t) * BN;
            const uint64_t dv = desc_add(dv0, static_cast<uint32_t>((s * C::V_STAGE) >> 4));
            const uint32_t first = (j > LEAD) ? 1u : 0u;  // the item's first PV overwrites O
            if (issuer) {
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk) {
                const uint64_t b = desc_add(dv, static_cast<uint32_t>((kk * 16 * 128) >> 4));
                mma_ts_one<C::MMA_CTAS>(tmem + C::O_COL, pcol + kk * 8, b, idesc_pv, kk == 0 ? first : 1u);
              }
            }
            __syncwarp();
            if constexpr (!C::MERGED_RELEASE) mma_commit_elect<C::MMA_CTAS>(&sb.v_empty[s]);
            mma_commit_elect<C::MMA_CTAS>(&sb.o_done[t & 1]);
          }
        }
        T += pl.n_tiles;
      }
      if (!ok && lane == 0) sb.wc.abort = 1;
      // All issued MMAs must finish before TMEM is released (and, in a pair,
      // before the peer's shared memory and TMEM go away).
      mma_commit_elect<C::MMA_CTAS>(&sb.final_mma);
      WaitCtl own_flag = own_wait_ctl(&sb.wc);
      mbar_wait(&sb.final_mma, 0, &own_flag, p.err, kDevTimeoutMma);
    } else if (warp == 1) {
      // A pair's rank 1: its TMEM is allocated by this warp; rank 0 issues the MMAs.
    } else if (warp == C::SCHED_WARP) {
      // ------------------------------------------------------------ scheduler
      // Finds this CTA's items, computes each valid item's geometry and
      // key-tile plan, and publishes them through the plan ring (up to
      // kPlanRing items ahead of the slowest consumer warp).  Items come from
      // a static stride and, for the last round, given a work-queue word, are
      // claimed one at a time from it.
      int n = 0;
      bool ok = true;
      auto publish = [&](const PlanEntry& e) -> bool {
        const int slot = n % kPlanRing;
        bool good = true;
        if (lane == 0 && n >= kPlanRing)
          good = mbar_wait(&sb.plan_empty[slot], ((n / kPlanRing) - 1) & 1, &sb.wc, p.err, kDevTimeoutOther);
        good = __shfl_sync(kFullMask, good, 0);
        if (good && lane == 0) {
          sb.plans[slot] = e;
          mbar_arrive(&sb.plan_full[slot]);  // release: the entry is visible to the waiting consumers
        }
        ++n;
        return good;
      };
      const int n_groups = gridDim.x / C::NCTA;  // clusters (single CTAs when NCTA == 1)
      // Items [0, n_static) are walked with a static stride, which keeps the
      // CTAs in lockstep on neighbouring items; the last kQueueRounds rounds
      // (all items when the stride leaves fewer) come from the work queue, so
      // that the tail goes to whichever CTA frees up first.  Without a queue
      // every item is static.
      //
      // Work queue: two 64-bit words, (launch tag << 32) | next item - n_static
      // and (launch tag << 32) | CTAs done.  The last claiming CTA to finish
      // resets the item counter to 0 under its tag, ready for the next launch
      // (a graph replay may carry the same tag).  A launch that finds another
      // tag (an uninitialised workspace, or one last used by another kernel)
      // installs its own with the counter at 1, taking the first queued item;
      // so the words need no initialisation.  Rank 0 claims entry c's item
      // once the producer has taken entry c - kClaimAhead (it starts loading an
      // item as the one before computes).  In a cluster of two, rank 1
      // receives each claim (or the end) through its claim slots.  Items
      // without rows are skipped by jumping to the next candidate
      // (next_candidate; in the queue by moving its counter with atomicMax).
      constexpr bool TWO = C::NCTA == 2;
      const bool dyn = p.queue != nullptr;
      // (kept in shared memory rather than a register: the control warps run
      // on a reduced register budget)
      if (lane == 0) sb.n_static = dyn ? max(0, n_items / n_groups - kQueueRounds) * n_groups : n_items;
      __syncwarp();
      const volatile int& n_static = sb.n_static;
      auto claim = [&](bool first) -> int {  // lane 0; first: this CTA's first claim
        const long long idx = queue_add(p.queue, first, p.err);
        return idx >= 0 && idx < n_items - n_static ? n_static + static_cast<int>(idx) : INT_MAX;
      };
      int item = -1;
      int round = -1;  // static rounds walked
      int qc = 0;  // claims made (rank 0) / received (rank 1)
      for (int c = 0; ok; ++c) {  // c: plan entries
        PlanEntry e;
        if (!dyn || item < n_static) {  // static phase
          // Round rr of the static rounds gives this CTA (group g) item
          // rr * n_groups + g.  When every item is static (no work queue),
          // odd rounds run backwards (rr * n_groups + n_groups - 1 - g): the
          // groups that take the first items of one round take the last of
          // the next, which evens out the items' costs across groups (they
          // fall with the position inside a (request, head) block).  Measured
          // on the windowed mixed batch's prefill rows: 0.588 vs 0.565 of the
          // bf16 peak; ahead of a queued last round it cost 1-5 %.
          const int g = blockIdx.x / C::NCTA;
          auto item_of = [&](long long rr) -> int {
            const long long it_ = rr * n_groups + ((!dyn && (rr & 1)) ? n_groups - 1 - g : g);
            return it_ >= n_items ? INT_MAX : static_cast<int>(it_);
          };
          ++round;
          item = item_of(round);
          while (item < n_static) {  // skip items without rows
            e.it = item_geometry<C, PAGED>(item, p);
            if (e.it.valid) break;
            const long long target = candidate_target<C>(item, e.it, p, lane);
            if (target >= n_items) {
              item = INT_MAX;
              break;
            }
            long long rr = target / n_groups;  // the first round whose item is at or after target
            if (static_cast<long long>(item_of(rr)) < target) ++rr;
            round = static_cast<int>(rr);
            item = item_of(round);
          }
        }
        if (dyn && item >= n_static) {  // queue phase
          const int slot = qc % kPlanRing;
          if (!TWO || rank == 0) {
            bool good = true;
            const int ct = c - kClaimAhead;  // entry the producer must have taken
            // (the producer cannot be past entry c - 1 here, and publishing
            // entry c - 1 needed entry c - 5 consumed, so the slot's phase
            // parity is exact)
            if (lane == 0 && ct >= 0)
              good = mbar_wait(&sb.plan_taken[ct % kPlanRing], (ct / kPlanRing) & 1, &sb.wc, p.err,
                               kDevTimeoutOther);
            if (lane == 0 && good) item = claim(qc == 0);
            ok = __shfl_sync(kFullMask, good, 0);
            item = __shfl_sync(kFullMask, item, 0);
            while (ok && item < n_items) {  // skip items without rows
              e.it = item_geometry<C, PAGED>(item, p);
              if (e.it.valid) break;
              const long long target = candidate_target<C>(item, e.it, p, lane);
              if (target >= n_items) {
                item = INT_MAX;
              } else {
                if (lane == 0) {
                  atomicMax(p.queue, (grid_launch_id() << 32) | static_cast<unsigned long long>(target - n_static));
                  item = claim(false);
                }
                item = __shfl_sync(kFullMask, item, 0);
              }
            }
            if constexpr (TWO) {
              if (lane == 0 && ok) {
                if (qc >= kPlanRing)
                  ok = mbar_wait_cluster(&sb.claim_empty[slot], ((qc / kPlanRing) - 1) & 1, &sb.wc, p.err,
                                         kDevTimeoutOther);
                if (ok) {
                  st_cluster_u32(mapa_shared(smem_u32(&sb.claims[slot]), 1), static_cast<uint32_t>(item));
                  mbar_arrive_cluster_release(mapa_shared(smem_u32(&sb.claim_full[slot]), 1));
                }
              }
              ok = __shfl_sync(kFullMask, ok, 0);
            }
          } else {
            if (lane == 0) {
              ok = mbar_wait_cluster(&sb.claim_full[slot], (qc / kPlanRing) & 1, &sb.wc, p.err,
                                     kDevTimeoutOther);
              if (ok) {
                item = sb.claims[slot];
                mbar_arrive_cluster_release(mapa_shared(smem_u32(&sb.claim_empty[slot]), 0));  // (after the read)
              }
            }
            ok = __shfl_sync(kFullMask, ok, 0);
            item = __shfl_sync(kFullMask, item, 0);
            if (ok && item < n_items) e.it = item_geometry<C, PAGED>(item, p);
          }
          ++qc;
        }
        if (!ok || item >= n_items) break;
        e.pl = plan_tiles<C>(e.it, p, use_table, lane);
        e.last = 0;
        ok = publish(e);
      }
      if (ok) {
        PlanEntry e{};
        e.last = 1;
        publish(e);
      }
    }
  } else if (warp < C::SOFTMAX_END) {
    // ------------------------------------------------------------ softmax rows
    if constexpr (C::REG_SPLIT) regs_increase<C::REGS_SOFTMAX>();
    constexpr int HC = C::HC;
    const int quarter = warp & 3;
    const int half = (warp - C::SOFTMAX_BEGIN) / 4;  // which column half of the row
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sc = p.m.scale_log2;  // > 0 (checked on the host)
    const bool key0_mode = p.m.sink_mode == 1 && p.m.sinks != nullptr;
    const bool null_mode = p.m.sink_mode == 2 && p.m.sinks != nullptr;
    float2* xslots = reinterpret_cast<float2*>(smem + C::RED_OFF);
    uint64_t* xb = sb.xchg[quarter];
    int xk = 0;  // exchanges done by this thread
    float2* rowinfo = reinterpret_cast<float2*>(smem + C::ROW_OFF);
    bool ok = true;
    int T = 0, n = 0, hk = 0;  // hk: items handed to the epilogue warps
    // This thread's row of an item: geometry, visible intervals and sink.
    struct RowCtx {
      int head, qi;
      bool valid;
      RowVis vis;
      float sink;
    };
    const int pos_off = row_pos_off();
    // p_full lives in rank 0: one arrival per warp (released at cluster scope in a pair)
    const uint32_t p_full_addr0 = C::PAIR ? mapa_shared(smem_u32(&sb.p_full[0]), 0) : 0u;
    // head-dim split: the peer's score buffer and barriers, and the exchanges done
    const uint32_t xs_peer = C::SPLITD ? mapa_shared(smem_u32(smem + C::XS_OFF), rank ^ 1) : 0u;
    const uint32_t x_full_peer = C::SPLITD ? mapa_shared(smem_u32(&sb.x_full[0]), rank ^ 1) : 0u;
    const uint32_t x_empty_peer = C::SPLITD ? mapa_shared(smem_u32(&sb.x_empty[0]), rank ^ 1) : 0u;
    int xs = 0, xr = 0;  // tiles of partial scores sent to / received from the peer
    // The row's global inputs (range-table entry, sink), loaded one item
    // ahead so that their latency hides behind the current item's tiles.
    struct RowLoads {
      int2 tab;
      float sink;
    };
    auto row_loads = [&](const PlanEntry& e) {
      RowLoads l;
      const int qi = e.it.pos0 + pos_off + row / p.gpack;
      const bool valid = !e.last && qi < e.it.q_len;
      l.tab = (valid && use_table) ? range_entry(p.m, e.it.q0 + qi, e.it.b, e.it.ctx + qi) : make_int2(1, 0);
      l.sink = (!e.last && p.m.sink_mode != 0 && p.m.sinks != nullptr) ? __ldg(p.m.sinks + e.it.h0 + (row % p.gpack))
                                                                       : 0.f;
      return l;
    };
    auto row_ctx = [&](const PlanEntry& e, const RowLoads& l) {
      RowCtx r;
      r.head = e.it.h0 + (row % p.gpack);
      r.qi = e.it.pos0 + pos_off + row / p.gpack;
      r.valid = !e.last && r.qi < e.it.q_len;
      r.vis = r.valid ? row_visibility_from(p.m, e.it.ctx + r.qi, e.it.k_len, use_table, l.tab) : empty_row();
      r.sink = l.sink;
      return r;
    };
    PlanEntry cur;
    ok = consume_plan(sb, n++, lane, cur, p.err);
    RowCtx rc = row_ctx(cur, row_loads(cur));
    while (ok && !cur.last) {
      // Take the next item's plan now and start its row loads; they are
      // used only after this item's tiles.
      PlanEntry nxt;
      if (ok) ok = consume_plan(sb, n++, lane, nxt, p.err);
      if (!ok) nxt.last = 1;
      const RowLoads nloads = row_loads(nxt);
      const Plan& pl = cur.pl;
      const RowVis vis = rc.vis;
      const float sink_l2 = rc.sink * 1.4426950408889634f;  // log2 units
      const float sink_raw = rc.sink / p.m.scale;            // units of the raw q.k score
      float m_ref = null_mode ? sink_l2 : -INFINITY;
      // Partial row sums of this thread's columns: the bf16-rounded
      // probabilities (they normalise O, which the PV MMA builds from them;
      // with ROWSUM the tensor core sums them and l_sum keeps only the null
      // logit's share) and the unrounded ones (they give the LSE).  The null
      // logit counts once.
      float l_sum = (null_mode && half == 0) ? 1.f : 0.f;
      float l_lse = l_sum;

      // A head-dim split runs one tile behind: step js sends tile js's
      // partial scores to the peer, then finishes tile js - 1, whose peer
      // partial has had a whole step to arrive.
      const int steps = pl.n_tiles + (C::SPLITD ? 1 : 0);
      for (int js = 0; js < steps; ++js) {
        if constexpr (C::SPLITD) {
          if (js < pl.n_tiles) {
            const int ts = T + js;
            if (!mbar_wait(&sb.s_full[ts & 1], (ts >> 1) & 1, &sb.wc, p.err, kDevTimeoutMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t ps[HC];
            const uint32_t pcol = tmem + lane_base + C::S_COL + (ts & 1) * BN;
#pragma unroll
            for (int c = 0; c < HC / 32; ++c)
              tmem_ld_32x32b_x32(pcol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&ps[c * 32]));
#pragma unroll
            for (int c = 0; c < HC / 32; ++c) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&ps[c * 32]));
            // the slot's previous tile (two back) must have been read by the peer
            const int slot = xs & 1;
            if (xs >= 2 &&
                !mbar_wait_cluster(&sb.x_empty[slot], ((xs - 2) >> 1) & 1, &sb.wc, p.err, kDevTimeoutSoftmax)) {
              ok = false;
              break;
            }
            const uint32_t dst = xs_peer + static_cast<uint32_t>(slot * kBM * BN * 4 + quarter * (BN / 4) * 512 + lane * 16);
#pragma unroll
            for (int c = 0; c < BN / 4; ++c)
              st_cluster_v4(dst + c * 512, ps[4 * c], ps[4 * c + 1], ps[4 * c + 2], ps[4 * c + 3]);
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_release(x_full_peer + slot * 8);
            ++xs;
          }
          if (js == 0) continue;
        }
        const int j = C::SPLITD ? js - 1 : js;
        const int t = T + j;
        const int kb = pl.kb_lo + j;
        const uint32_t scol = tmem + lane_base + C::S_COL + C::sbuf(t) * BN;
        if (!C::SPLITD && !mbar_wait(&sb.s_full[C::sbuf(t)], C::sphase(t), &sb.wc, p.err, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[HC];
#pragma unroll
        for (int c = 0; c < HC / 32; ++c)
          tmem_ld_32x32b_x32(scol + half * HC + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));

        if constexpr (C::SPLITD) {
          // The row's scores are the sum of both CTAs' partial products over
          // their halves of the head dimension: add the peer's partial of this
          // tile (sent a step ago) to this CTA's.  Both CTAs add the same two
          // fp32 values, so both go on with identical scores.  A slot holds,
          // per warp quarter and 4-score chunk, the 32 lanes' 16 bytes side by
          // side, so every warp-wide remote store and local load covers 512
          // contiguous bytes.
          const int slot = xr & 1;
          if (!mbar_wait_cluster(&sb.x_full[slot], (xr >> 1) & 1, &sb.wc, p.err, kDevTimeoutSoftmax)) {
            ok = false;
            break;
          }
          const uint4* src = reinterpret_cast<const uint4*>(smem + C::XS_OFF + slot * kBM * BN * 4 +
                                                            quarter * (BN / 4) * 512) + lane;
#pragma unroll
          for (int c = 0; c < BN / 4; ++c) {
            const uint4 v = src[c * 32];
            s[4 * c] = __float_as_uint(__uint_as_float(s[4 * c]) + __uint_as_float(v.x));
            s[4 * c + 1] = __float_as_uint(__uint_as_float(s[4 * c + 1]) + __uint_as_float(v.y));
            s[4 * c + 2] = __float_as_uint(__uint_as_float(s[4 * c + 2]) + __uint_as_float(v.z));
            s[4 * c + 3] = __float_as_uint(__uint_as_float(s[4 * c + 3]) + __uint_as_float(v.w));
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_release(x_empty_peer + slot * 8);
          ++xr;
        }

        // Mask: one bit per key of this thread's columns.  Scores stay in raw
        // q.k units; the scale folds into the exponent's FFMA (scale > 0).
        const bool masked = !(kb >= pl.int_lo && kb <= pl.int_hi) || (key0_mode && kb == 0);
        if (masked) {
          const int c0 = kb * BN + half * HC;  // first key of these columns
          if (key0_mode && c0 == 0 && vis.visible(0)) s[0] = __float_as_uint(__uint_as_float(s[0]) + sink_raw);
#pragma unroll
          for (int w = 0; w < HC / 32; ++w) {
            const uint32_t bits = interval_bits(vis.b_lo, vis.b_hi, c0 + 32 * w) |
                                  interval_bits(vis.r_lo, vis.r_hi, c0 + 32 * w);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              s[32 * w + i] = ((bits >> i) & 1u) ? s[32 * w + i] : __float_as_uint(-INFINITY);
          }
        }
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(s[k]), __uint_as_float(s[k + 8]));
#pragma unroll
        for (int i = 16; i < HC; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mx8[k] = fmax3(mx8[k], __uint_as_float(s[i + k]), __uint_as_float(s[i + 8 + k]));
        float mx_raw = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        if constexpr (C::SPLIT > 1) {
          // the two halves of a row meet once per tile
          float2 other;
          if (!pair_exchange(xslots, xb, xk, half, row, make_float2(mx_raw, 0.f), other, &sb.wc, p.err)) {
            ok = false;
            break;
          }
          mx_raw = fmaxf(mx_raw, other.x);
        }
        const float mx = mx_raw * sc;
        // lazy reference max
        float alpha = 1.f;
        const bool need = (mx > m_ref + kRescaleThreshold) || (m_ref == -INFINITY && mx > -INFINITY);
        if (need) {
          alpha = ex2_approx(m_ref - mx);  // 0 when m_ref == -inf
          l_sum *= alpha;
          l_lse *= alpha;
          m_ref = mx;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const uint64_t sc2 = f2_pack(sc, sc);
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t acc_e[4];
        float acc_lo[4], acc_hi[4];  // (MIXED_SUM: rounded probabilities of the even, odd columns)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc_e[k] = 0ull;
          acc_lo[k] = acc_hi[k] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < HC / 2; ++i) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), sc2, nm2), t0, t1);
          const float e0 = ex2_approx(t0);
          const float e1 = ex2_approx(t1);
          const uint32_t pk = pack_bf16x2(e0, e1);
          if constexpr (C::MIXED_SUM)  // (else the tensor core sums the rounded values)
            add_bf16x2_halves(pk, acc_lo[i & 3], acc_hi[i & 3]);
          if constexpr (LSE) acc_e[i & 3] = f2_add(acc_e[i & 3], f2_pack(e0, e1));
          s[i] = pk;
        }
        {
          float a0, a1, b0, b1;
          if constexpr (C::MIXED_SUM) {
            a0 = (acc_lo[0] + acc_lo[1]) + (acc_lo[2] + acc_lo[3]);
            a1 = (acc_hi[0] + acc_hi[1]) + (acc_hi[2] + acc_hi[3]);
            l_sum += a0 + a1;
          }
          if constexpr (LSE) {
            f2_unpack(f2_add(f2_add(acc_e[0], acc_e[1]), f2_add(acc_e[2], acc_e[3])), b0, b1);
            l_lse += b0 + b1;
          }
        }
        // P (bf16 pairs) over this half's scores.  Both halves have their
        // scores in registers (the exchange above), so neither overwrites
        // columns the other still has to read.
#pragma unroll
        for (int c = 0; c < HC / 64; ++c)
          tmem_st_32x32b_x32(scol + half * (HC / 2) + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&s[c * 32]));

        // O correction for rows whose reference moved (warp-uniform branch:
        // tcgen05.ld/st are warp-collective); each half corrects its columns.
        if (j > 0 && __any_sync(kFullMask, need)) {
          const int tp = t - 1;  // the previous tile's PV must have landed in O
          if (!mbar_wait(&sb.o_done[tp & 1], (tp >> 1) & 1, &sb.wc, p.err, kDevTimeoutMma)) ok = false;
          if (ok) {
            tc_fence_after();
            const uint32_t ocol = tmem + lane_base + C::O_COL + C::ocol(half * C::HDV);
#pragma unroll 1
            for (int c = 0; c < C::HDV / 32; ++c) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(ocol + c * 32, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
              tmem_st_32x32b_x32(ocol + c * 32, o);
            }
            if constexpr (C::ROWSUM) {
              if (half == 0) {  // the row sum (first of its equal columns) moves with O
                const uint32_t lcol = tmem + lane_base + C::L_COL;
                uint32_t lv = tmem_ld_32x32b_x1(lcol);
                tmem_ld_wait1(lv);
                tmem_st_32x32b_x1(lcol, __float_as_uint(__uint_as_float(lv) * alpha));
              }
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        // (fault injection for the timeout tests: one warp withholds the first
        // tile's arrival, so the MMA issuer's bounded wait runs out)
        const bool withhold = p.m.fault == kFaultWithholdProbs && T == 0 && j == 0 &&
                              warp == C::SOFTMAX_BEGIN && (C::NCTA == 1 || cluster_rank() == 0);
        if (lane == 0 && !withhold) {
          if constexpr (C::PAIR) mbar_arrive_cluster(p_full_addr0 + C::sbuf(t) * 8);
          else mbar_arrive(&sb.p_full[C::sbuf(t)]);
        }
        if (!ok) break;
      }

      // ---------------------------------------------------------- end of item
      const RowCtx nrc = row_ctx(nxt, nloads);
      if constexpr (C::SPLIT > 1) {
        // combine the halves' partial sums
        float2 other;
        if (ok && pair_exchange(xslots, xb, xk, half, row, make_float2(l_sum, l_lse), other, &sb.wc, p.err)) {
          l_sum += other.x;
          l_lse += other.y;
        } else {
          ok = false;
        }
      }
      // Hand the row's normaliser and LSE to the epilogue warps, which read
      // O out of TMEM once the item's last PV is done; these warps go on to
      // the next item at once.
      if (half == 0) {
        const int slot = hk % C::EPI_SLOTS;
        if (hk >= C::EPI_SLOTS &&
            !mbar_wait(&sb.epi_empty[slot], ((hk / C::EPI_SLOTS) - 1) & 1, &sb.wc, p.err, kDevTimeoutStore))
          ok = false;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // ROWSUM: the epilogue adds the tensor core's row sum to l_sum (then
        // the null logit's share alone) and inverts it
        const float inv_l = C::ROWSUM ? l_sum : ((l_sum > 0.f) ? 1.f / l_sum : 0.f);
        const float lse = (l_lse > 0.f) ? (m_use + lg2_approx(l_lse)) * 0.6931471805599453f : -INFINITY;
        rowinfo[slot * kBM + row] = make_float2(inv_l, lse);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.epi_full[slot]);  // release: the row values are visible
      }
      ++hk;
      T += pl.n_tiles;
      cur = nxt;
      rc = nrc;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    if constexpr (C::REG_SPLIT) regs_decrease<C::REGS_EPI>();
    // One thread per row (TMEM lane): waits for the row's (1 / l, LSE) from
    // the softmax warps and for the item's last PV, reads O out of TMEM 32
    // columns at a time, normalises, stores; after the last TMEM read it
    // releases O for the next item's first PV (o_free).
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int pos_off = row_pos_off();
    const bool out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
    const float2* rowinfo = reinterpret_cast<const float2*>(smem + C::ROW_OFF);
    const uint32_t o_free_addr0 = C::PAIR ? mapa_shared(smem_u32(&sb.o_free), 0) : 0u;
    const int oc0 = C::SPLITD ? rank * C::OC : 0;  // this CTA's first output column of the item
    bool ok = true;
    int T = 0, hk = 0;
    for (int n = 0; ok; ++n) {
      PlanEntry e;
      ok = consume_plan(sb, n, lane, e, p.err);
      if (!ok || e.last) break;
      const int head = e.it.h0 + (row % p.gpack);
      const int qi = e.it.pos0 + pos_off + row / p.gpack;
      const bool valid = qi < e.it.q_len && in_bounds(e.it.q0 + qi, p.total_q, p.err);  // (checked build)
      const int slot = hk % C::EPI_SLOTS;
      if (!mbar_wait(&sb.epi_full[slot], (hk / C::EPI_SLOTS) & 1, &sb.wc, p.err, kDevTimeoutSoftmax)) {
        ok = false;
        break;
      }
      const float2 info = rowinfo[slot * kBM + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.epi_empty[slot]);
      ++hk;
      const bool has_tiles = e.pl.n_tiles > 0;
      float inv_l = info.x;
      if (has_tiles) {
        const int tl = T + e.pl.n_tiles - 1;  // the item's last PV
        if (!mbar_wait(&sb.o_done[tl & 1], (tl >> 1) & 1, &sb.wc, p.err, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if constexpr (C::ROWSUM) {
        // the row's sum of bf16 probabilities (tensor core) + the null logit's share
        float l = info.x;
        if (has_tiles) {
          uint32_t lv = tmem_ld_32x32b_x1(tmem + lane_base + C::L_COL);
          tmem_ld_wait1(lv);
          l += __uint_as_float(lv);
        }
        inv_l = (l > 0.f) ? 1.f / l : 0.f;
      }
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                            (static_cast<size_t>(e.it.q0 + qi) * p.hq + head) * C::D + e.it.dv0 + oc0;
      const uint32_t ocol = tmem + lane_base + C::O_COL;
#pragma unroll 1
      for (int c = 0; c < C::OC / 32; ++c) {
        uint32_t o[32];
        if (has_tiles) {
          tmem_ld_32x32b_x32(ocol + C::ocol(c * 32), o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int v = 0; v < 32; ++v) o[v] = 0u;
        }
        if (has_tiles && c == C::OC / 32 - 1) {
          // O is out of TMEM: the next item's first PV may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (C::PAIR) mbar_arrive_cluster(o_free_addr0);
            else mbar_arrive(&sb.o_free);
          }
        }
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int v = 0; v < 16; ++v)
            w[v] = pack_bf16x2(__uint_as_float(o[2 * v]) * inv_l, __uint_as_float(o[2 * v + 1]) * inv_l);
          __nv_bfloat16* dst = orow + c * 32;
          if (out_v8) {
            st_global_v8(dst, w);
            st_global_v8(dst + 16, w + 8);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int v = 0; v < 4; ++v) d4[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
      }
      if (valid && p.lse != nullptr && e.it.dv0 == 0 && oc0 == 0)
        p.lse[static_cast<size_t>(head) * p.total_q + e.it.q0 + qi] = info.y;
      T += e.pl.n_tiles;
    }
    if (!ok && lane == 0) sb.wc.abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  // This CTA claims no more items (also after an abort): count it, and the
  // launch's last claiming CTA resets the work queue.
  // (The rank is read again: keeping it live through the roles costs registers.)
  if (p.queue != nullptr && threadIdx.x == C::SCHED_WARP * 32 && (C::NCTA == 1 || cluster_rank() == 0))
    queue_finish(p.queue, gridDim.x / C::NCTA, p.err);
  // a pair: rank 0's MMAs and drain are complete; a head-dim split: the peer
  // no longer writes into this CTA's shared memory
  if constexpr (C::NCTA == 2) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (C::PAIR) tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

using Cfg64 = Cfg<64, 64, 128, 4, 4, 1>;
// D = 128: the softmax warps bound the tile, so the tensor core also sums
// the rows (TMEM: 2 x 128 S + 160 accumulator columns; shared memory: two
// K and two V stages, each V stage with its ones block).
using Cfg128 = Cfg<128, 128, 128, 2, 2, 2, 0, 2, 1>;
using Cfg256 = Cfg<256, 256, 128, 2, 2, 2>;
// D = 512: O of all 512 value columns does not fit TMEM next to S, so the
// default splits the value dimension over two items (each recomputes S).  The
// alternative keeps O resident by splitting the head dimension over a 2-CTA
// cluster (no recomputation, partial scores exchanged every tile); it meets
// the same tolerances but measured slower on GB300 (the exchange and its
// cluster-scope release cost more per tile than the recomputed QK), so a
// caller selects it explicitly (the head-split variant of
// mvp_attn_fwd_varlen_ext).
using Cfg512 = Cfg<512, 256, 64, 2, 2, 2>;
using Cfg512S = Cfg<512, 512, 64, 2, 1, 2, 1>;

// Per-device launch state of one kernel instantiation: its dynamic shared
// memory attribute is set once, and the number of co-resident CTA pairs is
// queried once (clusters must fit within a GPC).  Guarded by a mutex: two host
// threads may make their first call on a device at the same time.
struct LaunchState {
  bool attr_set = false;
  int active_pairs = 0;
};
std::mutex g_launch_mutex;

template <class C>
cudaError_t launch_cfg(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       cudaStream_t stream) {
  const bool paged = p.m.block_table != nullptr;
  const bool want_lse = p.lse != nullptr;
  auto kern = paged ? (want_lse ? attn_prefill_kernel<C, true, true> : attn_prefill_kernel<C, true, false>)
                    : (want_lse ? attn_prefill_kernel<C, false, true> : attn_prefill_kernel<C, false, false>);
  static LaunchState state[4][64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  LaunchState& ls = state[(paged ? 1 : 0) + (want_lse ? 2 : 0)][dev];
  const long long n_items =
      static_cast<long long>(p.n_qtiles) * (p.num_reqs - p.req_offset) * p.hkv * p.n_hgroups * C::DV_SPLIT;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > INT_MAX) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::NCTA;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // (the occupancy query below sees the cluster shape only)
  // Persistent groups: as many CTAs (pairs) as can be resident at once.
  int groups = p.n_ctas / C::NCTA;
  {
    std::lock_guard<std::mutex> lock(g_launch_mutex);
    if (!ls.attr_set) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      ls.attr_set = true;
    }
    if (C::NCTA > 1 && ls.active_pairs == 0) {
      cfg.gridDim = dim3(groups * C::NCTA);
      int active = 0;
      e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
      if (e != cudaSuccess) return e;
      ls.active_pairs = active > 0 ? active : groups;
    }
  }
  if (C::NCTA > 1 && ls.active_pairs < groups) groups = ls.active_pairs;
  if (n_items < groups) groups = static_cast<int>(n_items);
  cfg.gridDim = dim3(groups * C::NCTA);
  cfg.numAttrs = 2;
  // Fewer than two rounds of items: every CTA takes at most two, the static
  // stride is as good, and the queue's atomics would only add latency.
  PrefillParams pq = p;
  if (n_items < 2LL * groups) pq.queue = nullptr;
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, pq);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

template <class C>
PrefillShape shape_of() {
  return {C::BN, C::DV, C::DV_SPLIT, C::BN, C::KROWS, C::NCTA, C::ITEM_ROWS, C::SPLITD ? 2 : 1, C::DQ, C::OC,
          C::ITEM_ROWS, C::OCW - C::OC};
}

PrefillShape prefill_tile_shape(int head_dim, bool d512_head_split) {
  switch (head_dim) {
    case 64: return shape_of<Cfg64>();
    case 128: return shape_of<Cfg128>();
    case 256: return shape_of<Cfg256>();
    case 512: return d512_head_split ? shape_of<Cfg512S>() : shape_of<Cfg512>();
    default: return {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
  }
}

cudaError_t launch_prefill(int head_dim, bool d512_head_split, const PrefillParams& p, const CUtensorMap& mq,
                           const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_cfg<Cfg64>(p, mq, mk, mv, stream);
    case 128: return launch_cfg<Cfg128>(p, mq, mk, mv, stream);
    case 256: return launch_cfg<Cfg256>(p, mq, mk, mv, stream);
    case 512:
      return d512_head_split ? launch_cfg<Cfg512S>(p, mq, mk, mv, stream) : launch_cfg<Cfg512>(p, mq, mk, mv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mvp
