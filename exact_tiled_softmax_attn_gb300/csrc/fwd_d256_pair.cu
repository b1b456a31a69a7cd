// bf16 attention forward for rows wider than 128 columns on CTA pairs (sm_103a).
//
// The same tiled online softmax as the one-CTA kernel in fwd_bf16_d256.cu
// ("Tiled attention with an online softmax", section "Task"; "The Hidden
// Recurrence in Softmax Attention", section "Chunk-wise Mode with Online
// Softmax Re-scale"), with a unit of two 128-row query tiles of one head, 2p
// and 2p + 1, computed by a cluster of two CTAs (rank c holds query tile
// 2p + c). Each product is one tcgen05 instruction with cta_group::2 (M = 256,
// each CTA's 128 rows in its own TMEM) whose B operand is split by its N
// columns between the two CTAs:
//   S = Q K^T  (A: this CTA's Q tile in shared memory)  B: CTA c holds keys [64c, 64c + 64) of the K tile
//   O += P V   (A: P in TMEM)                            B: CTA c holds columns [c dv/2, (c + 1) dv/2) of V
// so each SM loads, and its tensor core reads, half of every K and V tile
// (64 KB per key tile at dv = 256 instead of 128 KB), and the same ring of
// five 32 KB slots holds two and a half key tiles instead of one and a
// quarter. The pair runs over the key tiles of its later query tile; the
// earlier tile's softmax masks the one tile it does not see.
//
// Roles as in the one-CTA kernel: warp 0 lane 0 the producer (both CTAs),
// warp 1 the MMA issuer (the leader, rank 0; both CTAs' warp 1 allocate and
// free the TMEM pair), warps 4-7 the softmax group, one thread per row (both
// CTAs). Q and the K / V halves of both CTAs complete on the leader's
// barriers (TMA with cta_group::2), the softmax warps of both CTAs arrive on
// the leader's p_full (one arrival per warp), and the leader's commits arrive
// on the barriers of both CTAs. TMEM of each CTA: two score buffers of 128
// columns and the O accumulator, as in the one-CTA kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace fwd256p {

// D[tmem, both CTAs] (+)= A[smem, each CTA its own rows] * B[smem, split by N]
// (the shared-memory-A form of ptx::mma_ts_pair)
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

constexpr int BM = 128;                  // query rows per CTA
constexpr int BN = 128;                  // keys per tile
constexpr int HD = 256;                  // Q / K tile width
constexpr int QBOX = BM * 64 * 2;        // TMA box of 128 rows x 64 bf16 (Q, V)
constexpr int KBOX = 64 * 64 * 2;        // TMA box of 64 rows x 64 bf16 (this CTA's half of K)
constexpr float TAU = 8.0f;              // lazy-rescale threshold (log2 units)
constexpr int NUM_THREADS = 256;
constexpr uint32_t T_O = 256;            // TMEM column of the O accumulator
// Time (ns) a producer that gave up lets pass before its CTA leaves, so that
// copies it issued have landed (their completion is counted on the leader's
// barriers, which it cannot wait on).
constexpr uint64_t kPairSettleNs = 20000000ull;

template <int HV>
struct Cfg {
  static_assert(HV == 128 || HV == 256, "V tile width");
  static constexpr int VB = HV / 128;            // 64-column boxes of this CTA's half of V
  static constexpr int TILE_Q = BM * HD * 2;     // 64 KB
  static constexpr int ITEM_K = 64 * HD * 2;     // 32 KB: 64 keys x 256 columns
  static constexpr int ITEM_V = VB * QBOX;       // 128 keys x HV / 2 columns
  static constexpr int SLOT = ITEM_K;
  static constexpr int NSLOT = 5;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + TILE_Q;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * SLOT;
  // q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], pv_done, o_full, drain
  static constexpr int NBAR = 2 + 2 * NSLOT + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16(256, BN, false, false);   // N = 128 keys, 64 per CTA
  static constexpr uint32_t IDESC_PV = ptx::idesc_bf16(256, HV, false, true);   // N = dv, dv / 2 per CTA
  static constexpr uint32_t SOFTMAX_WARPS_PAIR = 8;                              // arrivals on p_full
};

struct Params {
  Problem p;
  __nv_bfloat16* O;
  float* LSE;
  uint32_t* status;
  UnitOrder order;   // units: (head, pair of 128-row query tiles)
  int n_kv_tiles;    // 128-key tiles
  int n_q_tiles;     // 128-row query tiles
  float sc2;         // scale * log2(e)
};

// Key tiles of the pair of query tiles 2 pq and 2 pq + 1: those of the later
// tile, or of the earlier one when the later lies past Tq.
__device__ __forceinline__ int pair_tiles(const Params& P, int pq) {
  const int last = min(2 * pq + 1, P.n_q_tiles - 1);
  return P.p.causal ? min(P.n_kv_tiles, last + 1) : P.n_kv_tiles;
}

template <int HV>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_d256_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK64,
                              const __grid_constant__ CUtensorMap tmV, const Params P) {
  using C = Cfg<HV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // (the same in both CTAs of a pair: both return, neither reaches a cluster barrier)
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  const uint32_t rank = ptx::cluster_ctarank();   // 0: leader, issues the pair's MMAs
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sKV = smem + C::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;               // leader's: both CTAs' Q tiles landed
  uint64_t* q_empty = bars + 1;              // the unit's last score product has read Q (both CTAs)
  uint64_t* kv_full = bars + 2;              // [NSLOT] leader's: both CTAs' halves of a K or V item landed
  uint64_t* kv_empty = kv_full + C::NSLOT;   // [NSLOT] the item's products are done (both CTAs)
  uint64_t* s_full = kv_empty + C::NSLOT;    // [2] by score buffer (both CTAs)
  uint64_t* p_full = s_full + 2;             // [2] leader's: both CTAs' P of the buffer is in TMEM
  uint64_t* pv_done = p_full + 2;            // one phase per P V product (both CTAs)
  uint64_t* o_full = pv_done + 1;            // the unit's last P V product is complete (both CTAs)
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
      ptx::mbar_init(p_full + b, C::SOFTMAX_WARPS_PAIR);
    }
    ptx::mbar_init(pv_done, 1);
    ptx::mbar_init(o_full, 1);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  // both CTAs' barriers are initialised before either signals the other's
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, 512);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_pairs = gridDim.x >> 1, pair = blockIdx.x >> 1;
  // Ring items (the same sequence in both CTAs), in the order the MMAs
  // consume them: K_0, K_1, then V_j followed by K_{j+2} for each j (a unit
  // of one tile: K_0, V_0); each item is this CTA's half of the tile. Item i
  // sits in slot i % NSLOT.
  auto slot = [](uint32_t item) { return static_cast<int>(item % C::NSLOT); };
  auto par = [](uint32_t item) { return (item / C::NSLOT) & 1u; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    ptx::WaitCtx w{abort_flag, P.status, 1u};
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK64);
    ptx::tma_prefetch_desc(&tmV);
    const uint32_t l_q_full = ptx::mapa_shared(ptx::smem_u32(q_full), 0);
    uint32_t item = 0, u_it = 0;
    bool ok = true;
    int bh, pq;
    for (int round = 0; ok && P.order.unit(pair, n_pairs, round, &bh, &pq); ++round) {
      const int nk = pair_tiles(P, pq);
      if (nk == 0) continue;
      // this CTA's query tile (rows past Tq read as zeros), counted on the
      // leader's q_full, which the leader's producer arms with both tiles
      if (!(ok = ptx::mbar_wait(q_empty, (u_it & 1u) ^ 1u, w))) break;
      if (rank == 0) ptx::mbar_arrive_expect_tx(q_full, 2 * C::TILE_Q);
      const int qrow = (2 * pq + static_cast<int>(rank)) * BM;
      for (int b = 0; b < HD / 64; ++b) ptx::tma_load_3d_pair(sQ + b * QBOX, &tmQ, l_q_full, b * 64, qrow, bh);
      auto load = [&](int kv, int j) {   // this CTA's half of K (kv = 0) or V (kv = 1) of key tile j
        const int sl = slot(item);
        if (!(ok = ptx::mbar_wait(kv_empty + sl, par(item) ^ 1u, w))) return;
        uint8_t* dst = sKV + sl * C::SLOT;
        const uint32_t mb = ptx::mapa_shared(ptx::smem_u32(kv_full + sl), 0);
        if (kv == 0) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(kv_full + sl, 2 * C::ITEM_K);
          for (int b = 0; b < HD / 64; ++b)
            ptx::tma_load_3d_pair(dst + b * KBOX, &tmK64, mb, b * 64, j * BN + 64 * static_cast<int>(rank), bh);
        } else {
          if (rank == 0) ptx::mbar_arrive_expect_tx(kv_full + sl, 2 * C::ITEM_V);
          for (int b = 0; b < C::VB; ++b)
            ptx::tma_load_3d_pair(dst + b * QBOX, &tmV, mb, static_cast<int>(rank) * (HV / 2) + b * 64, j * BN, bh);
        }
        ++item;
      };
      for (int j = 0; ok && j < 2 && j < nk; ++j) load(0, j);
      for (int j = 0; ok && j < nk; ++j) {
        load(1, j);
        if (ok && j + 2 < nk) load(0, j + 2);
      }
      ++u_it;
    }
    if (!ok) {
      // Copies in flight count on the leader's barriers; let them land
      // before this CTA can leave (the other roles give up within their bound).
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::globaltimer_ns() - t0 < kPairSettleNs) {
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (leader)
    // The whole warp follows the schedule; the elect.sync lane issues the
    // MMAs and commits (a commit tracks its own thread's MMAs).
    ptx::WaitCtx w{abort_flag, P.status, 3u};
    const uint32_t sQa = ptx::smem_u32(sQ), sKVa = ptx::smem_u32(sKV);
    // S_g = Q K_g^T into score buffer g & 1 of both CTAs: 16 k-steps over the
    // 256 columns, B = this CTA's 64 keys of the K item in slot sl
    auto mma_S = [&](uint32_t g, int sl) {
      const uint32_t d = tmem + 128 * (g & 1u);
      const uint64_t a0 = ptx::sdesc_sw128(sQa, 16, 1024);
      const uint64_t b0 = ptx::sdesc_sw128(sKVa + sl * C::SLOT, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        mma_ss_pair(d, ptx::sdesc_advance(a0, (kk >> 2) * QBOX + (kk & 3) * 32),
                         ptx::sdesc_advance(b0, (kk >> 2) * KBOX + (kk & 3) * 32), C::IDESC_S, kk > 0 ? 1u : 0u);
    };
    // O (+)= P_g V_g: 8 k-steps over the tile's 128 keys, B = this CTA's
    // dv / 2 columns of the V item in slot sl (MN-major, 64-column boxes)
    auto mma_PV = [&](uint32_t g, int sl, bool acc) {
      const uint32_t a = tmem + 128 * (g & 1u);   // P_g: bf16 pairs in the first 64 columns
      const uint64_t b0 = ptx::sdesc_sw128(sKVa + sl * C::SLOT, QBOX, 1024);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)
        ptx::mma_ts_pair(tmem + T_O, a + kk * 8, ptx::sdesc_advance(b0, kk * 2048), C::IDESC_PV,
                         (acc || kk > 0) ? 1u : 0u);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    uint32_t g0 = 0, u_it = 0;   // g0: global index of the unit's first key tile
    uint32_t item = 0;           // ring position, advanced in the producer's order
    bool ok = true, moved = false;
    int bh, pq;
    for (int round = 0; ok && P.order.unit(pair, n_pairs, round, &bh, &pq); ++round) {
      const int nk = pair_tiles(P, pq);
      if (nk == 0) continue;
      if (!(ok = wait(q_full, u_it & 1u))) break;
      // S_g from the K item at the ring position; its commit also completes
      // the score buffer (and, for the unit's last tile, the use of Q)
      auto issue_S = [&](uint32_t g, bool last_S) {
        const uint32_t ik = item++;
        if (!(ok = wait(kv_full + slot(ik), par(ik)))) return;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
          mma_S(g, slot(ik));
          ptx::mma_commit_pair(kv_empty + slot(ik));
          ptx::mma_commit_pair(s_full + (g & 1u));
          if (last_S) ptx::mma_commit_pair(q_empty);
        }
        __syncwarp();
      };
      // the scores of the first two key tiles
      for (int jj = 0; ok && jj < 2 && jj < nk; ++jj) issue_S(g0 + jj, jj + 1 == nk);
      if (!ok) break;
      for (int j = 0; j < nk; ++j) {
        const uint32_t g = g0 + j;
        if (!(ok = wait(p_full + (g & 1u), (g >> 1) & 1u))) break;
        const uint32_t iv = item++;
        if (!(ok = wait(kv_full + slot(iv), par(iv)))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
          mma_PV(g, slot(iv), j > 0);
          ptx::mma_commit_pair(kv_empty + slot(iv));
          ptx::mma_commit_pair(pv_done);
          if (j + 1 == nk) ptx::mma_commit_pair(o_full);
        }
        __syncwarp();
        // S_{g+2} into the buffer P_g V_g has just read (MMAs run in issue order)
        if (j + 2 < nk) issue_S(g + 2, j + 3 == nk);
        if (!ok) break;
      }
      if (!ok) break;
      g0 += nk;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit_pair(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax (both CTAs)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                    // row within this CTA's query tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + lane_off + T_O;
    ptx::WaitCtx w{abort_flag, P.status, 4u};
    const float sc2 = P.sc2;
    const int Tq = P.p.Tq, Tk = P.p.Tk;
    const int dv = P.p.dv;   // <= HV; a multiple of 8
    const uint32_t l_p_full0 = ptx::mapa_shared(ptx::smem_u32(p_full), 0);
    const uint32_t l_p_full1 = ptx::mapa_shared(ptx::smem_u32(p_full + 1), 0);
    uint32_t g0 = 0, u_it = 0;
    bool ok = true;
    int bh, pq;
    for (int round = 0; ok && P.order.unit(pair, n_pairs, round, &bh, &pq); ++round) {
      const int nk = pair_tiles(P, pq);
      if (nk == 0) continue;
      const int qt = 2 * pq + static_cast<int>(rank);
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
        const int kv0 = j * BN;
        if ((P.p.causal && kv0 + BN - 1 > qt * BM) || kv0 + BN > Tk) {
          // keys [0, lim) allowed; none for the earlier tile of the pair on
          // the later tile's last key tile
          const int lim = min(Tk - kv0, P.p.causal ? q_row - kv0 + 1 : BN);
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
        // one arrival per warp at the leader's p_full, after every lane's
        // TMEM stores are complete and fenced
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster((g & 1u) ? l_p_full1 : l_p_full0);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(o_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.0f / l : 0.f;
      const bool row_ok = q_row < Tq;
      const float lse_row = (l > 0.f) ? (m_used + log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
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
      // (the next unit's first P V product, which overwrites O, waits for
      // both CTAs' p_full of that unit, signalled after this)
      ptx::tc_fence_before();
      g0 += nk;
      ++u_it;
    }
  }

  // No CTA of the pair frees the TMEM pair or leaves while the other may still
  // signal its barriers or have its memory read by the leader's MMAs.
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

// Pairs resident at once on this device, per kernel instantiation (the SMs of
// a TPC run the two CTAs of a pair).
template <int HV>
cudaError_t max_pairs(int* out) {
  constexpr int kMaxDevices = 64;
  static int cached[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg<HV>::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, attn_fwd_d256_pair_kernel<HV>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    cached[dev] = n;
  }
  *out = cached[dev];
  return cudaSuccess;
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
  P.n_q_tiles = (a.p.Tq + BM - 1) / BM;
  const long long n_blocks = (P.n_q_tiles + 1) / 2;
  if (n_blocks * a.p.B * a.p.H > 0x7fffffffLL) return cudaErrorInvalidValue;
  P.order.n_blocks = static_cast<int>(n_blocks);
  P.order.n_heads = a.p.B * a.p.H;
  P.order.heavy_last = a.p.causal ? 1 : 0;
  P.sc2 = a.p.scale * 1.4426950408889634f;
  auto kern = attn_fwd_d256_pair_kernel<HV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int pairs = 0;
  if ((e = max_pairs<HV>(&pairs)) != cudaSuccess) return e;
  const int units = P.order.count();
  if (units < pairs) pairs = units;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *a.tmQ, *a.tmK, *a.tmV, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fwd256p

cudaError_t launch_fwd_bf16_d256_pair(const LaunchFwd& a) {
  // dv below the V tile width runs with zero columns
  return a.p.dv > 128 ? fwd256p::launch<256>(a) : fwd256p::launch<128>(a);
}

}  // namespace attn
