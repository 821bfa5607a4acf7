// Masked varlen attention forward, prefill rows: tcgen05 + TMA, sm_103a.
//
// Computes, for a 128-row query tile, softmax(scale * Q K^T + mask) V with the
// online (running max / running sum) formulation in base 2, as the Triton
// kernel of vLLM PR #49815 does ("Key source snippets", the sinks branch of
// _fwd_kernel: exp2 domain, sink * log2(e), null-logit init m = sink, l = 1, or
// key-0 bias added to the masked score of key 0).  The mask is the
// (causal AND window) OR range rule of vLLM PR #50294's mask_mod, evaluated as
// two closed key intervals per row (mask.cuh).
//
// GB300 design (not the pages' kernels):
// * One CTA = one 128-row tile.  With GQA, G_pack query heads of one KV head
//   share the tile: row r is (position r / G_pack, head h0 + r % G_pack), so a
//   K/V tile read from L2 serves G_pack heads.  The Q tile is a single 3-D TMA
//   box (64 dims, G_pack heads, 128 / G_pack positions), 128-byte swizzled.
// * Warp roles: warp 0 issues TMA loads, warp 1 allocates TMEM and issues
//   tcgen05.mma from one thread, and SPLIT softmax warpgroups (warps 2..)
//   own the rows: with BN = 128 two warpgroups split every row's 128 scores
//   into halves of 64 (warps w and w+4 read the same TMEM lanes), exchange
//   the row max through shared memory once per tile, and split the O
//   correction and epilogue by columns.  One thread handles 64 scores, so
//   the exp/sum work of a tile is spread over twice as many warps.
// * TMEM (512 columns): S double buffer [0, BN) and [BN, 2 BN) in fp32; the
//   bf16 probabilities P overwrite the first BN/2 columns of their S buffer and
//   feed O += P V as the TMEM operand of tcgen05.mma; O at [2 BN, 2 BN + DV).
// * MMA order per step j: S_j = Q K_j^T, then O += P_{j-1} V_{j-1}, so the
//   tensor core computes the next scores while the softmax warps work on the
//   current ones.
// * Key tiles are visited only inside [min hull, max hull] of the tile's rows;
//   tiles fully inside every row's all-visible interval skip the mask.
// * O is rescaled lazily: a row's reference max only moves when the new max
//   exceeds it by more than 2^8 (probabilities then stay <= 256), so O is read
//   and written back rarely.
// * Every barrier wait is bounded (ptx.cuh).
#include <cuda_bf16.h>

#include "mask.cuh"
#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {

namespace {

constexpr int kBM = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// KB: 64-dim K chunks released per barrier; VK: keys per V barrier chunk.
template <int D_, int DV_, int BN_, int KST_, int VST_, int KB_ = 1, int VK_ = 32>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int DV = DV_;        // value columns handled by one CTA
  static constexpr int BN = BN_;
  static constexpr int KST = KST_;
  static constexpr int VST = VST_;
  static constexpr int QCH = D / 64;            // 64-dim chunks of Q and K (one TMA box each)
  static constexpr int KB = KB_;
  static constexpr int KBC = QCH / KB;          // K barrier chunks per tile
  static constexpr int VCH = DV / 64;           // 64-dim chunks of a V tile
  static constexpr int VK = VK_;
  static constexpr int VKC = BN / VK;           // V barrier chunks per tile
  static constexpr int K_CHUNK_BYTES = BN * 128;
  static constexpr int V_KEYCHUNK_BYTES = VK * DV * 2;
  static constexpr int SPLIT = BN / 64;         // softmax warpgroups (column halves of a row)
  static constexpr int HC = BN / SPLIT;         // score columns per softmax thread (64)
  static constexpr int HDV = DV / SPLIT;        // O columns per softmax thread
  static constexpr int THREADS = 64 + 128 * SPLIT;
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int K_BYTES = BN * D * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_BYTES;
  static constexpr int V_OFF = K_OFF + KST * K_BYTES;
  static constexpr int TILE_BYTES = V_OFF + VST * V_BYTES;
  static constexpr int RED_OFF = TILE_BYTES;                       // row-max / row-sum exchange
  static constexpr int RED_BYTES = SPLIT > 1 ? 2 * SPLIT * kBM * 4 : 0;
  static constexpr int SMEM_BYTES = RED_OFF + RED_BYTES + 1024;  // + alignment slack
  static constexpr int S_COL = 0;
  static constexpr int O_COL = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(O_COL + DV <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
  static_assert(BN == 64 || BN == 128, "BN");
  static_assert(HDV % 32 == 0, "O columns per thread");
  static_assert(DV % 64 == 0 && DV <= 256, "DV");
  static_assert(KST >= 1 && KST <= 4 && VST >= 1 && VST <= 4, "stages");
  static_assert(KST * KBC <= 16 && VST * VKC <= 16, "barrier arrays");
  static_assert(QCH % KB == 0 && BN % VK == 0 && VK % 16 == 0, "chunking");
};

struct __align__(8) Barriers {
  uint64_t q_full;
  uint64_t k_full[16];   // [stage][64-dim chunk]
  uint64_t k_empty[16];
  uint64_t v_full[16];   // [stage][32-key chunk]
  uint64_t v_empty[16];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t final_mma;
  uint32_t tmem_base;
  int abort_flag;
  int red[4];  // min hull lo, max hull hi, max core lo, min core hi
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Barriers sb;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- tile
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);  // heavy (late) tiles first
  const int b = blockIdx.y + p.req_offset;
  const int dv_split = (C::DV < C::D) ? (C::D / C::DV) : 1;
  const int zz = blockIdx.z;
  const int dv0 = (zz % dv_split) * C::DV;
  const int hz = zz / dv_split;
  const int hkv = hz / p.n_hgroups;
  const int h0 = hkv * (p.hq / p.hkv) + (hz % p.n_hgroups) * p.gpack;

  const int q0 = __ldg(p.m.cu_q + b);
  const int q_len = __ldg(p.m.cu_q + b + 1) - q0;
  const int k0 = __ldg(p.m.cu_k + b);
  const int k_len = __ldg(p.m.cu_k + b + 1) - k0;
  const int bmp = kBM / p.gpack;  // positions per tile
  const int pos0 = qt * bmp;
  if (pos0 >= q_len) return;                  // uniform over the CTA
  if (p.skip_decode && q_len == 1) return;    // handled by the decode kernel
  const int ctx = p.m.ctx_lens ? __ldg(p.m.ctx_lens + b) : (k_len - q_len);
  const bool use_table = table_active(p.m);

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    mbar_init(&sb.q_full, 1);
    for (int i = 0; i < 16; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 128 * C::SPLIT);
      mbar_init(&sb.o_done[i], 1);
    }
    mbar_init(&sb.final_mma, 1);
    sb.abort_flag = 0;
    sb.red[0] = INT_MAX;
    sb.red[1] = INT_MIN;
    sb.red[2] = INT_MIN;
    sb.red[3] = INT_MAX;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&sb.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;

  // Q load does not depend on the key range: start it right away.
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    mbar_arrive_expect_tx(&sb.q_full, C::Q_BYTES);
    for (int c = 0; c < C::QCH; ++c)
      tma_load_3d(sQ + c * (kBM * 128), &map_q, &sb.q_full, c * 64, h0, q0 + pos0);
  }

  // Row geometry (softmax warps): interval reduction over the tile's rows.
  const bool is_softmax = warp >= 2;
  const int quarter = warp & 3;
  const int half = is_softmax ? (warp - 2) / 4 : 0;  // which column half of the row
  const int row = quarter * 32 + lane;
  const int rpos = row / p.gpack;
  const int head = h0 + (row % p.gpack);
  const int qi = pos0 + rpos;
  const bool row_valid = is_softmax && qi < q_len;
  const int qpos = ctx + qi;
  RowVis vis = empty_row();
  if (row_valid) {
    vis = row_visibility(p.m, qpos, k_len, use_table ? (q0 + qi) : -1);
  }
  if (row_valid && half == 0) {
    int hl, hh, cl, ch;
    vis.hull(hl, hh);
    vis.core(cl, ch);
    if (hl <= hh) {
      atomicMin(&sb.red[0], hl);
      atomicMax(&sb.red[1], hh);
    }
    atomicMax(&sb.red[2], cl);   // empty core (INT_MAX, INT_MIN) kills the interior
    atomicMin(&sb.red[3], ch);
  }
  __syncthreads();

  const int BN = C::BN;
  int kb_lo = 0, n_tiles = 0, int_lo = 1, int_hi = 0;
  if (sb.red[0] <= sb.red[1]) {
    kb_lo = sb.red[0] / BN;
    const int kb_hi = sb.red[1] / BN;
    n_tiles = kb_hi - kb_lo + 1;
    if (sb.red[2] <= sb.red[3]) {
      int_lo = (sb.red[2] + BN - 1) / BN;
      int_hi = (sb.red[3] + 1) / BN - 1;
    }
  }
  const bool key0_mode = p.m.sink_mode == 1 && p.m.sinks != nullptr;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Loads follow the MMA consumption order: K_0, then per step j K_{j+1}
    // and V_j.  K is released per 64-dim chunk (as the QK MMAs of that chunk
    // finish) and V per 32-key chunk (as the PV MMAs over those keys finish),
    // so the next tile streams in while the current one is still in use.
    if (lane == 0) {
      bool ok = true;
      int kc = 0, vc = 0;  // tiles issued
      int k_armed[16], v_armed[16];  // times each full barrier was armed
#pragma unroll
      for (int i = 0; i < 16; ++i) k_armed[i] = v_armed[i] = 0;
      auto load_k = [&](int j) -> bool {
        const int s = kc % C::KST;
        const int krow = k0 + (kb_lo + j) * BN;
        uint8_t* dst = sK + s * C::K_BYTES;
#pragma unroll
        for (int g = 0; g < C::KBC; ++g) {
          uint64_t* full = &sb.k_full[s * C::KBC + g];
          if (kc >= C::KST &&
              !mbar_wait(&sb.k_empty[s * C::KBC + g], ((kc / C::KST) - 1) & 1, &sb.abort_flag, p.err,
                         kDevTimeoutLoad))
            return false;
          mbar_arrive_expect_tx(full, C::KB * C::K_CHUNK_BYTES);
#pragma unroll
          for (int cc = 0; cc < C::KB; ++cc) {
            const int c = g * C::KB + cc;
            tma_load_3d(dst + c * C::K_CHUNK_BYTES, &map_k, full, c * 64, hkv, krow);
          }
          ++k_armed[s * C::KBC + g];
        }
        ++kc;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = vc % C::VST;
        const int krow = k0 + (kb_lo + j) * BN;
        uint8_t* dst = sV + s * C::V_BYTES;
#pragma unroll
        for (int q = 0; q < C::VKC; ++q) {
          uint64_t* full = &sb.v_full[s * C::VKC + q];
          if (vc >= C::VST &&
              !mbar_wait(&sb.v_empty[s * C::VKC + q], ((vc / C::VST) - 1) & 1, &sb.abort_flag, p.err,
                         kDevTimeoutLoad))
            return false;
          mbar_arrive_expect_tx(full, C::V_KEYCHUNK_BYTES);
#pragma unroll
          for (int c = 0; c < C::VCH; ++c)
            tma_load_3d(dst + c * (BN * 128) + q * C::VK * 128, &map_v, full, dv0 + c * 64, hkv, krow + q * C::VK);
          ++v_armed[s * C::VKC + q];
        }
        ++vc;
        return true;
      };
      if (n_tiles > 0) ok = load_k(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) ok = load_k(j + 1);
        if (ok) ok = load_v(j);
      }
      // Drain: never leave the CTA with a TMA write still in flight.  Each
      // full barrier's last armed phase is waited for; these waits ignore the
      // CTA abort flag (issued copies always complete, and they must before
      // the CTA exits).
      if (!ok) sb.abort_flag = 1;
      volatile int own_flag = 0;
      mbar_wait(&sb.q_full, 0, &own_flag, nullptr, 0);
      for (int i = 0; i < 16; ++i) {
        if (k_armed[i] > 0) mbar_wait(&sb.k_full[i], (k_armed[i] - 1) & 1, &own_flag, nullptr, 0);
        if (v_armed[i] > 0) mbar_wait(&sb.v_full[i], (v_armed[i] - 1) & 1, &own_flag, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every tcgen05.mma.  Descriptors are computed once;
    // inside the unrolled loops each MMA only adds a compile-time offset, so
    // the issue loop stays shorter than the tensor core's work.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, C::BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, C::DV, false, true);
      const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), BN * 128, 1024);
      bool ok = n_tiles > 0 ? mbar_wait(&sb.q_full, 0, &sb.abort_flag, p.err, kDevTimeoutLoad) : true;
      for (int j = 0; ok && j <= n_tiles; ++j) {
        if (j < n_tiles) {
          const int s = j % C::KST;
          const uint32_t d = tmem + C::S_COL + (j & 1) * BN;
          const uint64_t dk = dk0 + static_cast<uint64_t>((s * C::K_BYTES) >> 4);
#pragma unroll
          for (int g = 0; g < C::KBC; ++g) {
            // smem written by TMA and published by the mbarrier needs no
            // tcgen05 fence; only TMEM hand-offs between threads do.
            if (!mbar_wait(&sb.k_full[s * C::KBC + g], (j / C::KST) & 1, &sb.abort_flag, p.err, kDevTimeoutLoad)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int cc = 0; cc < C::KB; ++cc) {
              const int c = g * C::KB + cc;
#pragma unroll
              for (int k16 = 0; k16 < 4; ++k16) {
                const uint64_t a = dq + static_cast<uint64_t>((c * (kBM * 128) + k16 * 32) >> 4);
                const uint64_t b = dk + static_cast<uint64_t>((c * C::K_CHUNK_BYTES + k16 * 32) >> 4);
                mma_bf16_ss(d, a, b, idesc_qk, (c | k16) != 0 ? 1u : 0u);
              }
            }
            mma_commit(&sb.k_empty[s * C::KBC + g]);
          }
          if (!ok) break;
          mma_commit(&sb.s_full[j & 1]);
        }
        if (j >= 1) {
          const int i = j - 1;
          if (!mbar_wait(&sb.p_full[i & 1], (i >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutSoftmax)) { ok = false; break; }
          tc_fence_after();
          const int s = i % C::VST;
          const uint32_t pcol = tmem + C::S_COL + (i & 1) * BN;
          const uint64_t dv = dv0 + static_cast<uint64_t>((s * C::V_BYTES) >> 4);
          const uint32_t first = (i > 0) ? 1u : 0u;
#pragma unroll
          for (int q = 0; q < C::VKC; ++q) {
            if (!mbar_wait(&sb.v_full[s * C::VKC + q], (i / C::VST) & 1, &sb.abort_flag, p.err, kDevTimeoutLoad)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int h = 0; h < C::VK / 16; ++h) {
              const int kk = q * (C::VK / 16) + h;  // 16-key step
              const uint64_t b = dv + static_cast<uint64_t>((kk * 16 * 128) >> 4);
              mma_bf16_ts(tmem + C::O_COL, pcol + kk * 8, b, idesc_pv, (q == 0 && h == 0) ? first : 1u);
            }
            mma_commit(&sb.v_empty[s * C::VKC + q]);
          }
          if (!ok) break;
          mma_commit(&sb.o_done[i & 1]);
        }
      }
      if (!ok) sb.abort_flag = 1;
      // All issued MMAs must finish before TMEM is released.
      mma_commit(&sb.final_mma);
      volatile int own_flag = 0;
      mbar_wait(&sb.final_mma, 0, &own_flag, p.err, kDevTimeoutMma);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    constexpr int HC = C::HC;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sc = p.m.scale_log2;  // > 0 (checked on the host)
    float sink_l2 = 0.f, sink_raw = 0.f;
    if (p.m.sink_mode != 0 && p.m.sinks != nullptr) {
      const float sk = __ldg(p.m.sinks + head);
      sink_l2 = sk * 1.4426950408889634f;  // log2 units
      sink_raw = sk / p.m.scale;            // units of the raw q.k score
    }
    const bool null_mode = p.m.sink_mode == 2 && p.m.sinks != nullptr;
    float m_ref = null_mode ? sink_l2 : -INFINITY;
    // Partial row sums of this thread's columns: the bf16-rounded
    // probabilities (they normalise O, which the PV MMA builds from them) and
    // the unrounded ones (they give the LSE).  The null-logit term counts once.
    float l_sum = (null_mode && half == 0) ? 1.f : 0.f;
    float l_lse = l_sum;
    float* red = reinterpret_cast<float*>(smem + C::RED_OFF);  // [2 parity][SPLIT][128]
    bool ok = true;

    for (int j = 0; j < n_tiles; ++j) {
      const int kb = kb_lo + j;
      const uint32_t scol = tmem + lane_base + C::S_COL + (j & 1) * BN;
      if (!mbar_wait(&sb.s_full[j & 1], (j >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutMma)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[HC];
#pragma unroll
      for (int c = 0; c < HC / 32; ++c)
        tmem_ld_32x32b_x32(scol + half * HC + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
#pragma unroll
      for (int c = 0; c < HC / 32; ++c) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));

      // Mask: one bit per key of this thread's 64 columns.  Scores stay in raw
      // q.k units; the scale folds into the exponent's FFMA (scale > 0).
      const bool masked = !(kb >= int_lo && kb <= int_hi) || (key0_mode && kb == 0);
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
        // the two halves of a row meet once per tile (double-buffered by parity)
        float* slot = red + (j & 1) * (C::SPLIT * kBM);
        slot[half * kBM + row] = mx_raw;
        named_barrier(1 + quarter, 64);
        mx_raw = fmaxf(mx_raw, slot[(1 - half) * kBM + row]);
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
      uint64_t acc_r[4], acc_e[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) acc_r[k] = acc_e[k] = 0ull;
#pragma unroll
      for (int i = 0; i < HC / 2; ++i) {
        float t0, t1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), sc2, nm2), t0, t1);
        const float e0 = ex2_approx(t0);
        const float e1 = ex2_approx(t1);
        const uint32_t pk = pack_bf16x2(e0, e1);
        acc_r[i & 3] = f2_add(acc_r[i & 3], f2_pack(__uint_as_float(pk << 16), __uint_as_float(pk & 0xffff0000u)));
        acc_e[i & 3] = f2_add(acc_e[i & 3], f2_pack(e0, e1));
        s[i] = pk;
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(f2_add(f2_add(acc_r[0], acc_r[1]), f2_add(acc_r[2], acc_r[3])), a0, a1);
        f2_unpack(f2_add(f2_add(acc_e[0], acc_e[1]), f2_add(acc_e[2], acc_e[3])), b0, b1);
        l_sum += a0 + a1;
        l_lse += b0 + b1;
      }
      // P (bf16 pairs) over this half's scores: HC/2 columns.  Both halves
      // have their scores in registers (the exchange above), so neither can
      // overwrite columns the other still has to read.
#pragma unroll
      for (int c = 0; c < HC / 64; ++c)
        tmem_st_32x32b_x32(scol + half * (HC / 2) + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&s[c * 32]));

      // O correction for rows whose reference moved (warp-uniform branch:
      // tcgen05.ld/st are warp-collective); each half corrects its columns.
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        const int i = j - 1;  // PV_{j-1} must have landed in O
        if (!mbar_wait(&sb.o_done[i & 1], (i >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutMma)) { ok = false; }
        if (ok) {
          tc_fence_after();
          const uint32_t ocol = tmem + lane_base + C::O_COL + half * C::HDV;
#pragma unroll 1
          for (int c = 0; c < C::HDV / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(ocol + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
            tmem_st_32x32b_x32(ocol + c * 32, o);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sb.p_full[j & 1]);
      if (!ok) break;
    }

    // ---------------------------------------------------------- epilogue
    if constexpr (C::SPLIT > 1) {
      // Combine the halves' partial sums.  After the first barrier neither
      // half still reads the last tile's max slot, so both parity slots are
      // free: one carries l_sum, the other l_lse.
      float* sa = red + (n_tiles & 1) * (C::SPLIT * kBM);
      float* sb2 = red + ((n_tiles + 1) & 1) * (C::SPLIT * kBM);
      named_barrier(1 + quarter, 64);
      sa[half * kBM + row] = l_sum;
      sb2[half * kBM + row] = l_lse;
      named_barrier(1 + quarter, 64);
      l_sum += sa[(1 - half) * kBM + row];
      l_lse += sb2[(1 - half) * kBM + row];
    }
    bool have_o = ok && n_tiles > 0;
    if (have_o) {
      const int i = n_tiles - 1;
      have_o = mbar_wait(&sb.o_done[i & 1], (i >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutMma);
      tc_fence_after();
    }
    const float inv_l = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
    __nv_bfloat16* orow = nullptr;
    if (row_valid)
      orow = reinterpret_cast<__nv_bfloat16*>(p.out) + (static_cast<size_t>(q0 + qi) * p.hq + head) * C::D + dv0 +
             half * C::HDV;
    const uint32_t ocol = tmem + lane_base + C::O_COL + half * C::HDV;
#pragma unroll 1
    for (int c = 0; c < C::HDV / 32; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld_32x32b_x32(ocol + c * 32, o);
        tmem_ld_wait(o);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t] = 0u;
      }
      if (row_valid) {
        uint32_t packed[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          packed[t] = pack_bf16x2(__uint_as_float(o[2 * t]) * inv_l, __uint_as_float(o[2 * t + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          dst[t] = make_uint4(packed[4 * t], packed[4 * t + 1], packed[4 * t + 2], packed[4 * t + 3]);
      }
    }
    if (row_valid && half == 0 && p.lse != nullptr && dv0 == 0) {
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float lse = (l_lse > 0.f) ? (m_use + lg2_approx(l_lse)) * 0.6931471805599453f : -INFINITY;
      p.lse[static_cast<size_t>(head) * p.total_q + q0 + qi] = lse;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Whole-tile load barriers: every extra tcgen05.commit / mbarrier wait costs
// issue slots of the single MMA thread, and finer release granularity was
// measured slower on GB300.
using Cfg64 = Cfg<64, 64, 128, 4, 4, 1, 128>;
using Cfg128 = Cfg<128, 128, 128, 2, 2, 2, 128>;
using Cfg256 = Cfg<256, 256, 128, 1, 1, 4, 128>;
using Cfg512 = Cfg<512, 256, 64, 1, 1, 8, 64>;

template <class C>
cudaError_t launch_cfg(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       cudaStream_t stream) {
  auto kern = attn_prefill_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int dv_split = C::D / C::DV;
  dim3 grid(p.n_qtiles, p.num_reqs - p.req_offset, p.hkv * p.n_hgroups * dv_split);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

PrefillShape prefill_tile_shape(int head_dim) {
  switch (head_dim) {
    case 64: return {Cfg64::BN, Cfg64::DV, 1, Cfg64::VK};
    case 128: return {Cfg128::BN, Cfg128::DV, 1, Cfg128::VK};
    case 256: return {Cfg256::BN, Cfg256::DV, 1, Cfg256::VK};
    case 512: return {Cfg512::BN, Cfg512::DV, Cfg512::D / Cfg512::DV, Cfg512::VK};
    default: return {0, 0, 0, 0};
  }
}

cudaError_t launch_prefill(int head_dim, const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_cfg<Cfg64>(p, mq, mk, mv, stream);
    case 128: return launch_cfg<Cfg128>(p, mq, mk, mv, stream);
    case 256: return launch_cfg<Cfg256>(p, mq, mk, mv, stream);
    case 512: return launch_cfg<Cfg512>(p, mq, mk, mv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mvp
