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
//   tcgen05.mma from one thread, warps 2..5 own one query row per thread
//   (softmax, O correction, epilogue).
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

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D_, int DV_, int BN_, int KST_, int VST_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int DV = DV_;        // value columns handled by one CTA
  static constexpr int BN = BN_;
  static constexpr int KST = KST_;
  static constexpr int VST = VST_;
  static constexpr int QCH = D / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int K_BYTES = BN * D * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_BYTES;
  static constexpr int V_OFF = K_OFF + KST * K_BYTES;
  static constexpr int TILE_BYTES = V_OFF + VST * V_BYTES;
  static constexpr int SMEM_BYTES = TILE_BYTES + 1024;  // + alignment slack
  static constexpr int S_COL = 0;
  static constexpr int O_COL = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(O_COL + DV <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(DV % 64 == 0 && DV <= 256, "DV");
  static_assert(KST >= 1 && KST <= 4 && VST >= 1 && VST <= 4, "stages");
};

struct __align__(8) Barriers {
  uint64_t q_full;
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[4];
  uint64_t v_empty[4];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t final_mma;
  uint32_t tmem_base;
  int abort_flag;
  int red[4];  // min hull lo, max hull hi, max core lo, min core hi
};

template <class C>
__global__ void __launch_bounds__(kThreads, 1)
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
    for (int i = 0; i < 4; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 128);
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
  const int row = quarter * 32 + lane;
  const int rpos = row / p.gpack;
  const int head = h0 + (row % p.gpack);
  const int qi = pos0 + rpos;
  const bool row_valid = is_softmax && qi < q_len;
  const int qpos = ctx + qi;
  RowVis vis = empty_row();
  if (row_valid) {
    vis = row_visibility(p.m, qpos, k_len, use_table ? (q0 + qi) : -1);
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
    if (lane == 0) {
      bool ok = true;
      int kc = 0, vc = 0;  // tiles issued
      auto load_k = [&](int j) -> bool {
        const int s = kc % C::KST;
        if (kc >= C::KST) {
          if (!mbar_wait(&sb.k_empty[s], ((kc / C::KST) - 1) & 1, &sb.abort_flag, p.err, kDevTimeoutLoad))
            return false;
        }
        mbar_arrive_expect_tx(&sb.k_full[s], C::K_BYTES);
        uint8_t* dst = sK + s * C::K_BYTES;
        const int krow = k0 + (kb_lo + j) * BN;
        for (int c = 0; c < C::QCH; ++c) tma_load_3d(dst + c * (BN * 128), &map_k, &sb.k_full[s], c * 64, hkv, krow);
        ++kc;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = vc % C::VST;
        if (vc >= C::VST) {
          if (!mbar_wait(&sb.v_empty[s], ((vc / C::VST) - 1) & 1, &sb.abort_flag, p.err, kDevTimeoutLoad))
            return false;
        }
        mbar_arrive_expect_tx(&sb.v_full[s], C::V_BYTES);
        uint8_t* dst = sV + s * C::V_BYTES;
        const int krow = k0 + (kb_lo + j) * BN;
        for (int c = 0; c < C::VCH; ++c)
          tma_load_3d(dst + c * (BN * 128), &map_v, &sb.v_full[s], dv0 + c * 64, hkv, krow);
        ++vc;
        return true;
      };
      if (n_tiles > 0) ok = load_k(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) ok = load_k(j + 1);
        if (ok) ok = load_v(j);
      }
      // Drain: never leave the CTA with a TMA write still in flight.  These
      // waits ignore the CTA abort flag (a private flag instead): issued
      // copies always complete, and they must before the CTA exits.
      if (!ok) sb.abort_flag = 1;
      volatile int own_flag = 0;
      mbar_wait(&sb.q_full, 0, &own_flag, nullptr, 0);
      for (int s = 0; s < C::KST; ++s) {
        if (kc > s) {
          const int last = ((kc - 1 - s) / C::KST) * C::KST + s;
          mbar_wait(&sb.k_full[s], (last / C::KST) & 1, &own_flag, nullptr, 0);
        }
      }
      for (int s = 0; s < C::VST; ++s) {
        if (vc > s) {
          const int last = ((vc - 1 - s) / C::VST) * C::VST + s;
          mbar_wait(&sb.v_full[s], (last / C::VST) & 1, &own_flag, nullptr, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, C::BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, C::DV, false, true);
      bool ok = n_tiles > 0 ? mbar_wait(&sb.q_full, 0, &sb.abort_flag, p.err, kDevTimeoutLoad) : true;
      for (int j = 0; ok && j <= n_tiles; ++j) {
        if (j < n_tiles) {
          const int s = j % C::KST;
          if (!mbar_wait(&sb.k_full[s], (j / C::KST) & 1, &sb.abort_flag, p.err, kDevTimeoutLoad)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + C::S_COL + (j & 1) * BN;
          const uint32_t kbase = smem_u32(sK + s * C::K_BYTES);
          const uint32_t qbase = smem_u32(sQ);
#pragma unroll
          for (int c = 0; c < C::QCH; ++c) {
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16) {
              const uint64_t a = smem_desc_sw128(qbase + c * (kBM * 128) + k16 * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(kbase + c * (BN * 128) + k16 * 32, 16, 1024);
              mma_bf16_ss(d, a, bd, idesc_qk, (c | k16) != 0);
            }
          }
          mma_commit(&sb.k_empty[s]);
          mma_commit(&sb.s_full[j & 1]);
        }
        if (j >= 1) {
          const int i = j - 1;
          if (!mbar_wait(&sb.p_full[i & 1], (i >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutSoftmax)) { ok = false; break; }
          const int s = i % C::VST;
          if (!mbar_wait(&sb.v_full[s], (i / C::VST) & 1, &sb.abort_flag, p.err, kDevTimeoutLoad)) { ok = false; break; }
          tc_fence_after();
          const uint32_t pcol = tmem + C::S_COL + (i & 1) * BN;
          const uint32_t vbase = smem_u32(sV + s * C::V_BYTES);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(vbase + kk * 16 * 128, BN * 128, 1024);
            mma_bf16_ts(tmem + C::O_COL, pcol + kk * 8, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sb.v_empty[s]);
          mma_commit(&sb.o_done[i & 1]);
        }
      }
      // All issued MMAs must finish before TMEM is released.
      mma_commit(&sb.final_mma);
      volatile int own_flag = 0;
      mbar_wait(&sb.final_mma, 0, &own_flag, p.err, kDevTimeoutMma);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sc = p.m.scale_log2;
    float sink_l2 = 0.f;
    if (p.m.sink_mode != 0 && p.m.sinks != nullptr) sink_l2 = __ldg(p.m.sinks + head) * 1.4426950408889634f;
    const bool null_mode = p.m.sink_mode == 2 && p.m.sinks != nullptr;
    float m_ref = null_mode ? sink_l2 : -INFINITY;
    float l_sum = null_mode ? 1.f : 0.f;   // sum of the bf16-rounded p: normalises O
    float l_lse = l_sum;                   // sum of the fp32 p: gives the LSE
    bool ok = true;

    for (int j = 0; j < n_tiles; ++j) {
      const int kb = kb_lo + j;
      const uint32_t scol = tmem + lane_base + C::S_COL + (j & 1) * BN;
      if (!mbar_wait(&sb.s_full[j & 1], (j >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutMma)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[C::BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld_32x32b_x32(scol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));

      const bool masked = !(kb >= int_lo && kb <= int_hi) || (key0_mode && kb == 0);
      float mx = -INFINITY;
      if (masked) {
        const int key0 = kb * BN;
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int key = key0 + i;
          float x = __uint_as_float(s[i]) * sc;
          if (key0_mode && key == 0) x += sink_l2;
          x = vis.visible(key) ? x : -INFINITY;
          s[i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      } else {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const float x = __uint_as_float(s[i]) * sc;
          s[i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
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
      // O is normalised by the sum of the bf16-rounded probabilities that the
      // PV MMA consumes (numerator and denominator use the same weights); the
      // LSE uses the sum of the unrounded ones.
      float part = 0.f, part_exact = 0.f;
#pragma unroll
      for (int i = 0; i < BN / 2; ++i) {
        const float e0 = ex2_approx(__uint_as_float(s[2 * i]) - m_use);
        const float e1 = ex2_approx(__uint_as_float(s[2 * i + 1]) - m_use);
        const uint32_t pk = pack_bf16x2(e0, e1);
        part += __uint_as_float(pk << 16) + __uint_as_float(pk & 0xffff0000u);
        part_exact += e0 + e1;
        s[i] = pk;
      }
      l_sum += part;
      l_lse += part_exact;
#pragma unroll
      for (int c = 0; c < BN / 64; ++c)
        tmem_st_32x32b_x32(scol + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&s[c * 32]));

      // O correction for rows whose reference moved (warp-uniform branch:
      // tcgen05.ld/st are warp-collective).
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        const int i = j - 1;  // PV_{j-1} must have landed in O
        if (!mbar_wait(&sb.o_done[i & 1], (i >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutMma)) { ok = false; }
        if (ok) {
          tc_fence_after();
          const uint32_t ocol = tmem + lane_base + C::O_COL;
#pragma unroll 1
          for (int c = 0; c < C::DV / 32; ++c) {
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
    bool have_o = ok && n_tiles > 0;
    if (have_o) {
      const int i = n_tiles - 1;
      have_o = mbar_wait(&sb.o_done[i & 1], (i >> 1) & 1, &sb.abort_flag, p.err, kDevTimeoutMma);
      tc_fence_after();
    }
    const float inv_l = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
    __nv_bfloat16* orow = nullptr;
    if (row_valid)
      orow = reinterpret_cast<__nv_bfloat16*>(p.out) + (static_cast<size_t>(q0 + qi) * p.hq + head) * C::D + dv0;
    const uint32_t ocol = tmem + lane_base + C::O_COL;
#pragma unroll 1
    for (int c = 0; c < C::DV / 32; ++c) {
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
    if (row_valid && p.lse != nullptr && dv0 == 0) {
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

using Cfg64 = Cfg<64, 64, 128, 4, 4>;
using Cfg128 = Cfg<128, 128, 128, 2, 2>;
using Cfg256 = Cfg<256, 256, 128, 1, 1>;
using Cfg512 = Cfg<512, 256, 64, 1, 1>;

template <class C>
cudaError_t launch_cfg(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       cudaStream_t stream) {
  auto kern = attn_prefill_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int dv_split = C::D / C::DV;
  dim3 grid(p.n_qtiles, p.num_reqs - p.req_offset, p.hkv * p.n_hgroups * dv_split);
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

PrefillShape prefill_tile_shape(int head_dim) {
  switch (head_dim) {
    case 64: return {Cfg64::BN, Cfg64::DV, 1};
    case 128: return {Cfg128::BN, Cfg128::DV, 1};
    case 256: return {Cfg256::BN, Cfg256::DV, 1};
    case 512: return {Cfg512::BN, Cfg512::DV, Cfg512::D / Cfg512::DV};
    default: return {0, 0, 0};
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
