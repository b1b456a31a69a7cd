// bf16 attention forward for head size d = 256 on tcgen05 tensor cores (and
// for any row wider than 128 columns: d or dv up to 256, a multiple of 8; the
// tensor maps read the columns up to 256, or up to the V tile width of 64,
// 128 or 256, as zeros, and the epilogue writes the first dv columns).
//
// The same tiled online softmax as the d <= 128 forward ("Tiled attention with
// an online softmax", section "Task"; "The Hidden Recurrence in Softmax
// Attention", section "Chunk-wise Mode with Online Softmax Re-scale"), laid
// out for a 256-wide Q row: a 128 x 256 bf16 Q tile is 64 KB, so a unit is one
// 128-row query tile of one head (not two). Keys come in tiles of 128 so that
// the score product Q K^T has N = 128: with both operands in shared memory an
// N = 64 product is held back by the shared-memory reads of its A operand
// (about 63% of the tensor rate, against the full rate at N = 128). A K or V
// tile is 64 KB (dv = 256), so each streams through a ring of five 32 KB
// slots as two items: K by halves of d (two 128-row x 64-column boxes), V by
// halves of the key range (dv / 64 boxes of 64 rows). Each half is released
// as soon as the products that read it complete.
//
// Warp roles (8 warps): warp 0 lane 0 TMA producer; warp 1 MMA issuer (one
// elected lane) and TMEM owner; warps 2-3 idle; warps 4-7 the softmax group,
// one thread per query row.
// TMEM (512 columns allocated): two score buffers of 128 fp32 columns at 0
// and 128, so the product S_{j+2} = Q K_{j+2}^T is issued as soon as P_j V_j
// has read P_j out of its buffer while the softmax still works on S_{j+1};
// the accumulator O at [256, 256 + dv). P_j goes back over the first 64
// columns of its buffer as packed bf16 and is the A operand of P_j V_j.
// The lazy rescale of O (when the running max grows by more than TAU) waits
// for the previous P V product, which the score product alone no longer
// orders: every step past the first waits for that product's completion.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace fwd256 {

constexpr int BM = 128;                  // query rows per unit
constexpr int BN = 128;                  // keys per tile
constexpr int HD = 256;                  // Q / K head size
constexpr int QBOX = BM * 64 * 2;        // TMA box of Q: 128 rows x 64 bf16
constexpr int KBOX = BN * 64 * 2;        // TMA box of K: 128 rows x 64 bf16
constexpr int VBOX = 64 * 64 * 2;        // TMA box of V: 64 rows x 64 bf16
constexpr float TAU = 8.0f;              // lazy-rescale threshold (log2 units)
constexpr int NUM_THREADS = 256;
constexpr uint32_t T_O = 256;            // TMEM column of the O accumulator

template <int HV>
struct Cfg {
  static constexpr int VB = HV / 64;             // 64-column boxes per V row
  static constexpr int TILE_Q = BM * HD * 2;     // 64 KB
  static constexpr int ITEM_K = 2 * KBOX;        // half of d of a K tile: 32 KB
  static constexpr int ITEM_V = VB * VBOX;       // half of the keys of a V tile: <= 32 KB
  static constexpr int SLOT = ITEM_K;
  static constexpr int NSLOT = 5;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + TILE_Q;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * SLOT;
  // q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], pv_done, o_full, drain
  static constexpr int NBAR = 2 + 2 * NSLOT + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16(BM, BN, false, false);
  static constexpr uint32_t IDESC_PV = ptx::idesc_bf16(BM, HV, false, true);
};

struct Params {
  Problem p;
  __nv_bfloat16* O;
  float* LSE;
  uint32_t* status;
  UnitOrder order;   // units: (head, 128-row query tile [, key range])
  int n_kv_tiles;    // 128-key tiles
  float sc2;         // scale * log2(e)
  // Split-KV mode (n_splits > 1): key range s of a query tile covers key
  // tiles [s * split_tiles, (s + 1) * split_tiles) and writes its normalised
  // partial output and log-sum-exp (fp32) to Opart [n_splits][B*H*Tq][dv]
  // and LSEpart [n_splits][B*H*Tq] instead of O and LSE.
  int n_splits;
  int split_tiles;
  float* Opart;
  float* LSEpart;
};

// 128-key tiles that query tile qt sees.
__device__ __forceinline__ int tiles_of(const Params& P, int qt) {
  return P.p.causal ? min(P.n_kv_tiles, qt + 1) : P.n_kv_tiles;
}

// Work unit `blk`: query tile qt, key range sp, first key tile j0 and tile
// count nk. nk = 0 for a range that starts past the query tile's last key
// tile (causal): no role touches such a unit and the merge never reads it.
template <bool SPLIT>
__device__ __forceinline__ void unit_range(const Params& P, int blk, int* qt, int* sp, int* j0, int* nk) {
  if (!SPLIT) {
    *qt = blk;
    *sp = 0;
    *j0 = 0;
    *nk = tiles_of(P, blk);
    return;
  }
  *qt = blk / P.n_splits;
  *sp = blk - *qt * P.n_splits;
  *j0 = *sp * P.split_tiles;
  *nk = max(0, min(tiles_of(P, *qt) - *j0, P.split_tiles));
}

template <int HV, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params P) {
  using C = Cfg<HV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sKV = smem + C::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;              // [NSLOT]
  uint64_t* kv_empty = kv_full + C::NSLOT;   // [NSLOT]
  uint64_t* s_full = kv_empty + C::NSLOT;    // [2], by score buffer
  uint64_t* p_full = s_full + 2;             // [2]
  uint64_t* pv_done = p_full + 2;            // one phase per P V product
  uint64_t* o_full = pv_done + 1;            // the unit's last P V product is complete
  uint64_t* drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(kv_full + s, 1);
      ptx::mbar_init(kv_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(s_full + b, 1);
      ptx::mbar_init(p_full + b, 128);
    }
    ptx::mbar_init(pv_done, 1);
    ptx::mbar_init(o_full, 1);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int grid = gridDim.x, cta = blockIdx.x;
  // Ring items, in the order the MMAs consume them: K_0, K_1, then V_j
  // followed by K_{j+2} for each j (a unit of one tile: K_0, V_0); every
  // tile is two items (K: d columns [0, 128) then [128, 256); V: keys
  // [0, 64) then [64, 128) of the tile). Item i sits in slot i % NSLOT.
  auto slot = [](uint32_t item) { return static_cast<int>(item % C::NSLOT); };
  auto par = [](uint32_t item) { return (item / C::NSLOT) & 1u; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::WaitCtx w{abort_flag, P.status, 1u};
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
    uint32_t item = 0, u_it = 0, q_issued = 0;   // q_issued: Q loads issued (one per unit)
    bool ok = true;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &blk); ++round) {
      int qt, sp, j0, nk;
      unit_range<SPLIT>(P, blk, &qt, &sp, &j0, &nk);
      if (nk == 0) continue;
      if (!(ok = ptx::mbar_wait(q_empty, (u_it & 1u) ^ 1u, w))) break;
      ptx::mbar_arrive_expect_tx(q_full, C::TILE_Q);
      for (int b = 0; b < HD / 64; ++b) ptx::tma_load_3d(sQ + b * QBOX, &tmQ, q_full, b * 64, qt * BM, bh);
      q_issued = u_it + 1;
      auto load = [&](int kv, int j) {   // both halves of K (kv = 0) or V (kv = 1) of key tile j
        for (int h = 0; ok && h < 2; ++h) {
          const int sl = slot(item);
          if (!(ok = ptx::mbar_wait(kv_empty + sl, par(item) ^ 1u, w))) return;
          uint8_t* dst = sKV + sl * C::SLOT;
          if (kv == 0) {
            ptx::mbar_arrive_expect_tx(kv_full + sl, C::ITEM_K);
            for (int b = 0; b < 2; ++b)
              ptx::tma_load_3d(dst + b * KBOX, &tmK, kv_full + sl, (2 * h + b) * 64, (j0 + j) * BN, bh);
          } else {
            ptx::mbar_arrive_expect_tx(kv_full + sl, C::ITEM_V);
            for (int b = 0; b < C::VB; ++b)
              ptx::tma_load_3d(dst + b * VBOX, &tmV, kv_full + sl, b * 64, (j0 + j) * BN + h * 64, bh);
          }
          ++item;
        }
      };
      for (int j = 0; ok && j < 2 && j < nk; ++j) load(0, j);
      for (int j = 0; ok && j < nk; ++j) {
        load(1, j);
        if (ok && j + 2 < nk) load(0, j + 2);
      }
      ++u_it;
    }
    if (!ok) {
      // Let the copies already in flight land before the CTA exits.
      for (uint32_t n = (item > (uint32_t)C::NSLOT ? item - C::NSLOT : 0u); n < item; ++n)
        ptx::mbar_wait_drain(kv_full + slot(n), par(n));
      // the last Q load issued (possibly this unit's, still in flight)
      if (q_issued > 0) ptx::mbar_wait_drain(q_full, (q_issued - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp follows the schedule; the elect.sync lane (lane 0)
    // issues the MMAs and commits (a commit tracks its own thread's MMAs).
    ptx::WaitCtx w{abort_flag, P.status, 3u};
    const uint32_t sQa = ptx::smem_u32(sQ), sKVa = ptx::smem_u32(sKV);
    // half h of S_g = Q K_g^T (d columns [128 h, 128 h + 128)) into score
    // buffer g & 1, from the K item in slot sl
    auto mma_S = [&](uint32_t g, int h, int sl) {
      const uint32_t d = tmem + 128 * (g & 1u);
      const uint64_t a0 = ptx::sdesc_sw128(sQa, 16, 1024);
      const uint64_t b0 = ptx::sdesc_sw128(sKVa + sl * C::SLOT, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_ss(d, ptx::sdesc_advance(a0, (2 * h + (kk >> 2)) * QBOX + (kk & 3) * 32),
                    ptx::sdesc_advance(b0, (kk >> 2) * KBOX + (kk & 3) * 32), C::IDESC_S,
                    (h > 0 || kk > 0) ? 1u : 0u);
    };
    // half h of O (+)= P_g V_g (keys [64 h, 64 h + 64) of the tile), from the
    // V item in slot sl
    auto mma_PV = [&](uint32_t g, int h, int sl, bool acc) {
      const uint32_t a = tmem + 128 * (g & 1u) + 32 * h;   // P_g: bf16 pairs in the first 64 columns
      const uint64_t b0 = ptx::sdesc_sw128(sKVa + sl * C::SLOT, VBOX, 1024);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ptx::mma_ts(tmem + T_O, a + kk * 8, ptx::sdesc_advance(b0, kk * 2048), C::IDESC_PV,
                    (acc || h > 0 || kk > 0) ? 1u : 0u);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    uint32_t g0 = 0, u_it = 0;   // g0: global index of the unit's first key tile
    uint32_t item = 0;           // ring position, advanced in the producer's order
    bool ok = true, moved = false;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &blk); ++round) {
      int qt, sp, j0, nk;
      unit_range<SPLIT>(P, blk, &qt, &sp, &j0, &nk);
      if (nk == 0) continue;
      if (!(ok = wait(q_full, u_it & 1u))) break;
      // S_g in two halves, each released as soon as it has been read; the
      // second half also completes the score buffer (and, for the unit's
      // last tile, its use of Q)
      auto issue_S = [&](uint32_t g, bool last_S) {
        for (int h = 0; h < 2; ++h) {
          const uint32_t ik = item++;
          if (!(ok = wait(kv_full + slot(ik), par(ik)))) return;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_S(g, h, slot(ik));
            ptx::mma_commit(kv_empty + slot(ik));
            if (h == 1) {
              ptx::mma_commit(s_full + (g & 1u));
              if (last_S) ptx::mma_commit(q_empty);
            }
          }
          __syncwarp();
        }
      };
      // the scores of the first two key tiles
      for (int jj = 0; ok && jj < 2 && jj < nk; ++jj) issue_S(g0 + jj, jj + 1 == nk);
      if (!ok) break;
      for (int j = 0; j < nk; ++j) {
        const uint32_t g = g0 + j;
        if (!(ok = wait(p_full + (g & 1u), (g >> 1) & 1u))) break;
        for (int h = 0; ok && h < 2; ++h) {
          const uint32_t iv = item++;
          if (!(ok = wait(kv_full + slot(iv), par(iv)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_PV(g, h, slot(iv), j > 0);
            ptx::mma_commit(kv_empty + slot(iv));
            if (h == 1) {
              ptx::mma_commit(pv_done);
              if (j + 1 == nk) ptx::mma_commit(o_full);
            }
          }
          __syncwarp();
        }
        if (!ok) break;
        // S_{g+2} into the buffer P_g V_g has just read (MMAs run in issue order)
        if (j + 2 < nk) issue_S(g + 2, j + 3 == nk);
        if (!ok) break;
      }
      if (!ok) break;
      g0 += nk;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                    // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + lane_off + T_O;
    ptx::WaitCtx w{abort_flag, P.status, 4u};
    const float sc2 = P.sc2;
    const int Tq = P.p.Tq, Tk = P.p.Tk;
    const int dv = P.p.dv;   // <= HV; a multiple of 8
    uint32_t g0 = 0, u_it = 0;
    bool ok = true;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &blk); ++round) {
      int qt, sp, j0, nk;
      unit_range<SPLIT>(P, blk, &qt, &sp, &j0, &nk);
      if (nk == 0) continue;
      const int q_row = qt * BM + r;
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < nk; ++j) {
        const uint32_t g = g0 + j;
        const uint32_t tS = tmem + lane_off + 128 * (g & 1u);
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(s_full + (g & 1u), (g >> 1) & 1u, w)))) break;
        ptx::tc_fence_after();
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, raw[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld_wait(raw[c]);
        float* s = reinterpret_cast<float*>(&raw[0][0]);
        const int kv0 = (j0 + j) * BN;
        if ((P.p.causal && kv0 + BN - 1 > qt * BM) || kv0 + BN > Tk) {
          const int lim = min(Tk - kv0, P.p.causal ? q_row - kv0 + 1 : BN);   // keys [0, lim) allowed
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (i >= lim) s[i] = -CUDART_INF_F;
        }
        float m4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmaxf(s[k], s[k + 4]);
#pragma unroll
        for (int i = 8; i < BN; i += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = ptx::fmax3(m4[k], s[i + k], s[i + 4 + k]);
        const float mx = ptx::fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sc2;
        const float m_new = fmaxf(m_used, mx);
        bool need = false;
        float corr = 1.0f;
        if (j == 0) {
          m_used = m_new;
        } else if (m_new > m_used + TAU) {
          need = true;
          corr = ptx::ex2(m_used - m_new);   // 0 when m_used = -inf
          l *= corr;
          m_used = m_new;
        }
        const float ref = (m_used == -CUDART_INF_F) ? 0.f : m_used;   // the -inf rule
        const float2 sc2v = make_float2(sc2, sc2), nrefv = make_float2(-ref, -ref);
        float2 ls[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ls[k] = make_float2(0.f, 0.f);
        // P over the first 64 columns of the buffer, 32 at a time (the scores
        // of both halves are already in registers)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = 64 * hh + 2 * i;
            const float2 x = ptx::ffma2(make_float2(s[c], s[c + 1]), sc2v, nrefv);
            const float2 pp = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            ls[i & 3] = ptx::fadd2(ls[i & 3], pp);
            pk[i] = ptx::pack_bf16(pp.x, pp.y);
          }
          ptx::tmem_st32(tS + 32 * hh, pk);
        }
        l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
        if (j > 0) {
          // the previous P V product is complete before O is rescaled (and
          // before the next one is released by p_full)
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(pv_done, (g - 1) & 1u, w)))) break;
          ptx::tc_fence_after();
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
            for (int c = 0; c < HV / 32; ++c) {
              uint32_t o[32];
              ptx::tmem_ld32(tO + c * 32, o);
              ptx::tmem_ld_wait(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
              ptx::tmem_st32(tO + c * 32, o);
            }
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full + (g & 1u));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(o_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.0f / l : 0.f;
      const bool row_ok = q_row < Tq;
      const float lse_row = (l > 0.f) ? (m_used + log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
      if (SPLIT) {
        // partial result of this key range: O_s = A / l in fp32 and LSE_s
        const size_t rows = static_cast<size_t>(P.p.B) * P.p.H * Tq;
        const size_t row = static_cast<size_t>(sp) * rows + static_cast<size_t>(bh) * Tq + (row_ok ? q_row : 0);
        float* prow = P.Opart + row * dv;
#pragma unroll 1
        for (int c = 0; c < HV / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + c * 32, o);
          ptx::tmem_ld_wait(o);
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(prow + c * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (c * 32 + 4 * v < dv)   // dv < HV: the padded columns stay unwritten
                dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                     __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
          }
        }
        if (row_ok) P.LSEpart[row] = lse_row;
        ptx::tc_fence_before();
        g0 += nk;
        ++u_it;
        continue;
      }
      __nv_bfloat16* orow = P.O + (static_cast<size_t>(bh) * Tq + (row_ok ? q_row : 0)) * dv;
#pragma unroll
      for (int c = 0; c < HV / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c * 32, o);
        ptx::tmem_ld_wait(o);
        uint32_t ob[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          ob[i] = ptx::pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (c * 32 + 8 * v < dv)   // dv < HV: the padded columns stay unwritten
              dst[v] = make_uint4(ob[4 * v], ob[4 * v + 1], ob[4 * v + 2], ob[4 * v + 3]);
        }
      }
      if (row_ok) P.LSE[static_cast<size_t>(bh) * Tq + q_row] = lse_row;
      ptx::tc_fence_before();
      g0 += nk;
      ++u_it;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int HV>
cudaError_t launch(const LaunchFwd& a) {
  using C = Cfg<HV>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory");
  Params P;
  P.p = a.p;
  P.O = reinterpret_cast<__nv_bfloat16*>(a.O);
  P.LSE = a.LSE;
  P.status = a.status;
  P.n_kv_tiles = (a.p.Tk + BN - 1) / BN;
  P.n_splits = a.n_splits > 1 ? a.n_splits : 1;
  P.split_tiles = a.split_tiles;
  P.Opart = a.Opart;
  P.LSEpart = a.LSEpart;
  const long long n_blocks = static_cast<long long>((a.p.Tq + BM - 1) / BM) * P.n_splits;
  if (n_blocks * a.p.B * a.p.H > 0x7fffffffLL) return cudaErrorInvalidValue;
  P.order.n_blocks = static_cast<int>(n_blocks);
  P.order.n_heads = a.p.B * a.p.H;
  P.order.heavy_last = a.p.causal ? 1 : 0;
  P.sc2 = a.p.scale * 1.4426950408889634f;
  const int units = P.order.count();
  const int grid = units < a.num_sms ? units : a.num_sms;
  auto kern = P.n_splits > 1 ? attn_fwd_d256_kernel<HV, true> : attn_fwd_d256_kernel<HV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, NUM_THREADS, C::SMEM, a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, P);
  return cudaGetLastError();
}

}  // namespace fwd256

cudaError_t launch_fwd_bf16_d256(const LaunchFwd& a) {
  // d below 256 and dv below the V tile width run with zero columns
  if (a.p.dv > 128) return fwd256::launch<256>(a);
  if (a.p.dv > 64) return fwd256::launch<128>(a);
  return fwd256::launch<64>(a);
}

}  // namespace attn
