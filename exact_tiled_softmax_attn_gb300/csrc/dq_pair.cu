// Deterministic dQ of the bf16 backward for d = 128 on CTA pairs (sm_103a).
//
// The same arithmetic as the one-CTA dQ kernel in bwd_bf16.cu ("attention_backprop",
// sections "Gradient of S" and "Gradient of Q and K"; P recomputed from the
// stored log-sum-exp as in "The Hidden Recurrence in Softmax Attention",
// section "Flash Attention Backward Pass"):
//   S = Q K^T, P = exp(scale S - LSE), dP = dO V^T, dS = P o (dP - D),
//   dQ = scale * sum over key tiles of dS K, in a fixed key order,
// but a unit is a pair of 128-row query tiles of one head, 2p and 2p + 1,
// computed by a cluster of two CTAs (rank c holds query tile 2p + c). One
// tcgen05 instruction with cta_group::2 then computes the products of both
// query tiles at once (M = 256, each CTA's rows in its own TMEM), and the B
// operand of each product is split by its N columns between the two CTAs:
//   S  = Q K^T  (A: Q in TMEM)   B = K rows:   CTA c holds keys [64c, 64c + 64) of the tile
//   dP = dO V^T (A: dO in TMEM)  B = V rows:   CTA c holds keys [64c, 64c + 64)
//   dQ += dS K  (A: dS in TMEM)  B = K columns: CTA c holds columns [64c, 64c + 64) of d
// so each CTA loads and its tensor core reads half of every K and V tile
// (48 KB per key tile instead of 64 KB loaded and 96 KB read), and each K or
// V tile is fetched from L2 once for two query tiles.
//
// The leader CTA (cluster rank 0) issues every MMA; its producer, the peer's
// producer and the row threads of both CTAs synchronise on the leader's
// mbarriers: the K and V halves of both CTAs complete on the leader's barrier
// (TMA with cta_group::2), the row threads of both CTAs arrive on it (one
// arrival per warp, at cluster scope), and the leader's commits arrive on
// both CTAs' barriers at once (multicast).
//
// Per CTA, warps: 0 producer (lane 0), 1 MMA issuer (rank 0 only; both CTAs'
// warp 1 allocate and free the TMEM pair), 2-5 and 6-9 the row groups as in
// the one-CTA kernel. Shared memory is one FIFO ring of 16 KB slots: per unit
// the two 64-row halves of this CTA's Q, dO and O tiles (the row threads
// move Q and dO into TMEM and form D = rowsum(dO o O), then release them),
// then per key tile: K_h (this CTA's 64 keys, all of d, the B operand of S),
// K_c (all 128 keys, this CTA's 64 columns of d, the B operand of dQ) and
// V_h (this CTA's 64 keys of V).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "bwd_common.cuh"
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace bwd {

template <int HV>
struct CfgP {
  static constexpr int HD = 128;
  static constexpr int BOX64 = 64 * 64 * 2;                 // one TMA box of 64 rows x 64 bf16
  static constexpr int SLOT = 16384;
  static constexpr uint32_t Q_HALF_BYTES = 64 * HD * 2;     // 64 query rows of Q
  static constexpr uint32_t V_HALF_BYTES = 64 * HV * 2;     // 64 rows of dO, O or V
  static constexpr uint32_t KH_BYTES = 64 * HD * 2;         // 64 keys of K, all of d
  static constexpr uint32_t KC_BYTES = 128 * 64 * 2;        // 128 keys of K, 64 columns of d
  static constexpr int DPART_BYTES = 2 * 2 * BT * 4;        // [unit parity][row group][128] fp32
  static constexpr int NSLOT = (227 * 1024 - DPART_BYTES - 512) / SLOT;   // 14
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_DPART = OFF_RING + NSLOT * SLOT;
  static constexpr int OFF_BAR = OFF_DPART + DPART_BYTES;
  // empty[NSLOT], kv_full[NSLOT], stg_full[NSLOT], stage_done, qd_ready, s_full, s_free, dp_full,
  // ds_full, dq_full, drain, dpart_full
  static constexpr int NBAR = 3 * NSLOT + 9;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16(256, BT, false, false);   // S, dP: N = 128 keys
  static constexpr uint32_t IDESC_DQ = ptx::idesc_bf16(256, HD, false, true);   // dQ: N = d, K MN-major
  // TMEM columns (the same in both CTAs)
  static constexpr uint32_t T_Q = 0, T_DO = 64, T_S = 128, T_DP = 256, T_DQ = 384;
  // arrivals at the leader's qd_ready, s_free and ds_full: one per row warp of both CTAs
  static constexpr uint32_t ROW_WARPS_PAIR = 16;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NSLOT <= 32, "per-slot phase bits");
};

// Pair unit `blk` of a head: query tiles 2 pq and 2 pq + 1, key split s, first
// key tile j0 and key tile count nk (the larger of the two tiles' counts: the
// first tile's rows mask the key tile it cannot see).
template <bool SPLIT>
__device__ __forceinline__ bool dq_pair_unit(const Params& P, int blk, int* pq, int* s, int* j0, int* nk) {
  const int S = SPLIT ? P.dq_splits : 1;
  *pq = SPLIT ? blk / S : blk;
  *s = SPLIT ? blk - *pq * S : 0;
  const int n = P.p.causal ? min(2 * *pq + 2, P.n_k_tiles) : P.n_k_tiles;
  *j0 = SPLIT ? *s * P.dq_split_tiles : 0;
  *nk = SPLIT ? max(0, min(n - *j0, P.dq_split_tiles)) : n;
  return *nk > 0;
}

// Time (ns) a producer that gave up lets pass before its CTA leaves, so that
// copies it issued have landed (their completion may be counted on the other
// CTA's barrier, which it cannot wait on).
constexpr uint64_t kPairSettleNs = 20000000ull;

template <int HV, bool SPLIT>
__global__ void __launch_bounds__(DQ_PAIR_THREADS, 1)
    dq_pair_kernel(const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ CUtensorMap tmK64,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV64,
                   const __grid_constant__ CUtensorMap tmdO64, const __grid_constant__ CUtensorMap tmO64,
                   const Params P) {
  using C = CfgP<HV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // (the same in both CTAs of a pair: both return, neither reaches a cluster barrier)
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  const uint32_t rank = ptx::cluster_ctarank();   // 0: leader, issues the pair's MMAs
  uint8_t* ring = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = bars;                    // [NSLOT] a slot's item has been consumed (both CTAs)
  uint64_t* kv_full = empty + C::NSLOT;      // [NSLOT] K / V halves of both CTAs landed (leader's)
  uint64_t* stg_full = kv_full + C::NSLOT;   // [NSLOT] this CTA's Q / dO / O half landed
  uint64_t* stage_done = stg_full + C::NSLOT;   // this CTA's row threads are done with the unit's staging slots
  uint64_t* qd_ready = stage_done + 1;       // leader's: Q and dO of both CTAs are in TMEM
  uint64_t* s_full = stage_done + 2;
  uint64_t* s_free = stage_done + 3;         // leader's: both CTAs' rows hold S in registers
  uint64_t* dp_full = stage_done + 4;
  uint64_t* ds_full = stage_done + 5;        // leader's: both CTAs' dS are in TMEM
  uint64_t* dq_full = stage_done + 6;
  uint64_t* drain = stage_done + 7;
  uint64_t* dpart_full = stage_done + 8;     // both row groups of this CTA wrote a unit's partial D
  float* dpart = reinterpret_cast<float*>(smem + C::OFF_DPART);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(empty + s, 1);
      ptx::mbar_init(kv_full + s, 1);
      ptx::mbar_init(stg_full + s, 1);
    }
    ptx::mbar_init(stage_done, 256);
    ptx::mbar_init(qd_ready, C::ROW_WARPS_PAIR);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_free, C::ROW_WARPS_PAIR);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(ds_full, C::ROW_WARPS_PAIR);
    ptx::mbar_init(dq_full, 1);
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(dpart_full, 256);
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
  const int Tq = P.p.Tq, Tk = P.p.Tk;
  // Ring item i (counted across units; the same sequence in both CTAs) sits
  // in slot i % NSLOT. A unit whose first item is i0 has the halves of Q at
  // i0, i0 + 1, of dO at i0 + 2, i0 + 3, of O at i0 + 4, i0 + 5, and K_h, K_c,
  // V_h of its j-th key tile at i0 + 6 + 3j, i0 + 7 + 3j, i0 + 8 + 3j.
  auto slot = [](uint32_t i) { return static_cast<int>(i % C::NSLOT); };
  auto par = [](uint32_t i) { return (i / C::NSLOT) & 1u; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    ptx::WaitCtx w{abort_flag, P.status, 17u};
    ptx::tma_prefetch_desc(&tmQ64);
    ptx::tma_prefetch_desc(&tmK64);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV64);
    ptx::tma_prefetch_desc(&tmdO64);
    ptx::tma_prefetch_desc(&tmO64);
    uint32_t item = 0;
    bool ok = true;
    int bh, blk;
    // a half of this CTA's Q, dO or O tile, counted on this CTA's barrier
    auto stage_load = [&](const CUtensorMap* map, int boxes, uint32_t bytes, int row) {
      const int s = slot(item);
      if (!ptx::mbar_wait(empty + s, par(item) ^ 1u, w)) return false;
      ptx::mbar_arrive_expect_tx(stg_full + s, bytes);
      for (int b = 0; b < boxes; ++b)
        ptx::tma_load_3d(ring + s * C::SLOT + b * C::BOX64, map, stg_full + s, b * 64, row, bh);
      ++item;
      return true;
    };
    // this CTA's half of a K or V tile, counted on the leader's barrier, which
    // the leader's producer arms with both CTAs' bytes
    auto kv_load = [&](const CUtensorMap* map, int boxes, int box_bytes, uint32_t bytes, int col0, int row) {
      const int s = slot(item);
      if (!ptx::mbar_wait(empty + s, par(item) ^ 1u, w)) return false;
      if (rank == 0) ptx::mbar_arrive_expect_tx(kv_full + s, 2 * bytes);
      const uint32_t mb = ptx::mapa_shared(ptx::smem_u32(kv_full + s), 0);
      for (int b = 0; b < boxes; ++b)
        ptx::tma_load_3d_pair(ring + s * C::SLOT + b * box_bytes, map, mb, col0 + b * 64, row, bh);
      ++item;
      return true;
    };
    for (int round = 0; ok && P.order.unit(pair, n_pairs, round, &bh, &blk); ++round) {
      int pq, sp_, j0, nk;
      if (!dq_pair_unit<SPLIT>(P, blk, &pq, &sp_, &j0, &nk)) continue;
      const int qrow = (2 * pq + static_cast<int>(rank)) * BT;   // this CTA's query tile (rows past Tq read as 0)
      for (int h = 0; ok && h < 2; ++h) ok = stage_load(&tmQ64, 2, C::Q_HALF_BYTES, qrow + 64 * h);
      for (int h = 0; ok && h < 2; ++h) ok = stage_load(&tmdO64, HV / 64, C::V_HALF_BYTES, qrow + 64 * h);
      for (int h = 0; ok && h < 2; ++h) ok = stage_load(&tmO64, HV / 64, C::V_HALF_BYTES, qrow + 64 * h);
      for (int j = 0; ok && j < nk; ++j) {
        const int kt = (j0 + j) * BT;
        ok = kv_load(&tmK64, 2, C::BOX64, C::KH_BYTES, 0, kt + 64 * static_cast<int>(rank)) &&
             kv_load(&tmK, 1, BOX_BYTES, C::KC_BYTES, 64 * static_cast<int>(rank), kt) &&
             kv_load(&tmV64, HV / 64, C::BOX64, C::V_HALF_BYTES, 0, kt + 64 * static_cast<int>(rank));
      }
    }
    if (!ok) {
      // Copies in flight may count on the leader's barriers; let them land
      // before this CTA can leave (the other roles give up within their bound).
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::globaltimer_ns() - t0 < kPairSettleNs) {
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (leader)
    ptx::WaitCtx w{abort_flag, P.status, 18u};
    const uint32_t aR = ptx::smem_u32(ring);
    auto kmaj64 = [](uint32_t base, int kk) {   // K-major B of 64 rows per CTA, k-step kk of 16 elements
      return ptx::sdesc_advance(ptx::sdesc_sw128(base, 16, 1024), (kk >> 2) * C::BOX64 + (kk & 3) * 32);
    };
    auto mnmaj = [](uint32_t base, int kk) {    // MN-major B (64 columns per CTA), k-step kk of 16 rows
      return ptx::sdesc_advance(ptx::sdesc_sw128(base, BOX_BYTES, 1024), kk * 2048);
    };
    auto waitc = [&](uint64_t* bar, uint32_t parity) {   // arrived at by both CTAs' row warps
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    uint32_t kvph = 0;   // per-slot phase bits of kv_full (only K / V items use it)
    auto wait_kv = [&](uint32_t it) {
      const int s = slot(it);
      const bool r = __all_sync(0xffffffffu, ptx::mbar_wait(kv_full + s, (kvph >> s) & 1u, w));
      kvph ^= 1u << s;
      return r;
    };
    auto mma_s = [&](uint32_t ih) {   // S = Q K^T; K_h of item ih is read by nothing later
#pragma unroll
      for (int kk = 0; kk < C::HD / 16; ++kk)
        ptx::mma_ts_pair(tmem + C::T_S, tmem + C::T_Q + 8 * kk, kmaj64(aR + slot(ih) * C::SLOT, kk), C::IDESC_S,
                         kk > 0);
      ptx::mma_commit_pair(s_full);
      ptx::mma_commit_pair(empty + slot(ih));
    };
    auto mma_dp = [&](uint32_t iv) {   // dP = dO V^T; V_h of item iv is read by nothing later
#pragma unroll
      for (int kk = 0; kk < HV / 16; ++kk)
        ptx::mma_ts_pair(tmem + C::T_DP, tmem + C::T_DO + 8 * kk, kmaj64(aR + slot(iv) * C::SLOT, kk), C::IDESC_S,
                         kk > 0);
      ptx::mma_commit_pair(dp_full);
      ptx::mma_commit_pair(empty + slot(iv));
    };
    uint32_t item = 0, u_it = 0, sp = 0;
    bool ok = true, moved = false;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(pair, n_pairs, round, &bh, &blk); ++round) {
      int pq, sp_, j0, nk;
      if (!dq_pair_unit<SPLIT>(P, blk, &pq, &sp_, &j0, &nk)) continue;
      const uint32_t i0 = item;
      if (!(ok = waitc(qd_ready, u_it & 1u))) break;
      // S and dP of the first key tile
      if (!(ok = wait_kv(i0 + 6))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        mma_s(i0 + 6);
      }
      __syncwarp();
      if (!(ok = wait_kv(i0 + 8))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        mma_dp(i0 + 8);
      }
      __syncwarp();
      if (nk > 1 && !(ok = wait_kv(i0 + 9))) break;
      for (int j = 0; j < nk; ++j, ++sp) {
        const uint32_t ih = i0 + 6 + 3 * j;   // K_h of tile j; K_c = ih + 1; V_h = ih + 2; tile j + 1 at ih + 3
        if (j + 1 < nk) {
          if (!(ok = waitc(s_free, sp & 1u))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_s(ih + 3);
          }
          __syncwarp();
        }
        // dQ += dS K
        if (!(ok = waitc(ds_full, sp & 1u))) break;
        if (!(ok = wait_kv(ih + 1))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)
            ptx::mma_ts_pair(tmem + C::T_DQ, tmem + C::T_DP + packed_col(kk), mnmaj(aR + slot(ih + 1) * C::SLOT, kk),
                             C::IDESC_DQ, (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit_pair(empty + slot(ih + 1));
        }
        __syncwarp();
        if (j + 1 < nk) {
          // dP of the next key tile, into the tile dQ_j has just been given
          if (!(ok = wait_kv(ih + 5))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_dp(ih + 5);
          }
          __syncwarp();
        }
        if (j + 2 < nk && !(ok = wait_kv(ih + 6))) break;
      }
      if (!ok) break;
      if (ptx::elect_one()) {
        moved |= lane != 0;
        ptx::mma_commit_pair(dq_full);
      }
      __syncwarp();
      item = i0 + 6 + 3 * nk;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit_pair(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ row groups (both CTAs)
    const int g = (warp - 2) >> 2;          // row group: key columns [64g, 64g + 64)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S + 64 * g, tDP = tmem + lane_off + C::T_DP + 64 * g;
    const uint32_t tDQ = tmem + lane_off + C::T_DQ + (C::HD / 2) * g;
    const uint32_t tQ = tmem + lane_off + C::T_Q + (C::HD / 4) * g, tDO = tmem + lane_off + C::T_DO + (HV / 4) * g;
    ptx::WaitCtx w{abort_flag, P.status, 19u + g};
    const float sc2 = P.sc2, scale = P.p.scale;
    const uint32_t l_qd_ready = ptx::mapa_shared(ptx::smem_u32(qd_ready), 0);
    const uint32_t l_s_free = ptx::mapa_shared(ptx::smem_u32(s_free), 0);
    const uint32_t l_ds_full = ptx::mapa_shared(ptx::smem_u32(ds_full), 0);
    // one arrival per warp at a barrier of the leader, after every lane's
    // TMEM accesses are complete and fenced
    auto warp_arrive_leader = [&](uint32_t cluster_addr) {
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(cluster_addr);
    };
    uint32_t stph = 0;   // per-slot phase bits of stg_full (only staging items use it)
    // Stage the unit whose first ring item is i0 (the u-th unit of this CTA):
    // this group's half of row r of Q and of dO into TMEM, its half of D_r =
    // sum_c dO_rc O_rc ("attention_backprop", section "Gradient of S") into
    // dpart, then give the six staging slots back. Rows past Tq load as zeros.
    auto stage = [&](uint32_t i0, uint32_t u) {
      for (int k = 0; k < 6; ++k) {
        const int s = slot(i0 + k);
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(stg_full + s, (stph >> s) & 1u, w))) return false;
        stph ^= 1u << s;
      }
      const int rl = r & 63, hf = r >> 6;   // row within its 64-row half
      const uint8_t* sq = ring + slot(i0 + hf) * C::SLOT;
      const uint8_t* sdo = ring + slot(i0 + 2 + hf) * C::SLOT;
      const uint8_t* so = ring + slot(i0 + 4 + hf) * C::SLOT;
      {
        uint32_t v[C::HD / 4];
#pragma unroll
        for (int k = 0; k < C::HD / 16; ++k) {
          const uint4 x = *reinterpret_cast<const uint4*>(sq + sw128_offset64(rl, (C::HD / 2) * g + 8 * k));
          v[4 * k] = x.x;
          v[4 * k + 1] = x.y;
          v[4 * k + 2] = x.z;
          v[4 * k + 3] = x.w;
        }
        ptx::tmem_st32(tQ, v);
      }
      float part = 0.f;
      {
        uint32_t v[HV / 4];
#pragma unroll
        for (int k = 0; k < HV / 16; ++k) {
          const uint32_t off = sw128_offset64(rl, (HV / 2) * g + 8 * k);
          const uint4 x = *reinterpret_cast<const uint4*>(sdo + off);
          const uint4 o = *reinterpret_cast<const uint4*>(so + off);
          v[4 * k] = x.x;
          v[4 * k + 1] = x.y;
          v[4 * k + 2] = x.z;
          v[4 * k + 3] = x.w;
          const __nv_bfloat162* dv = reinterpret_cast<const __nv_bfloat162*>(&x);
          const __nv_bfloat162* ov = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = __bfloat1622float2(ov[e]), b = __bfloat1622float2(dv[e]);
            part = fmaf(a.x, b.x, part);
            part = fmaf(a.y, b.y, part);
          }
        }
        if constexpr (HV == 128) ptx::tmem_st32(tDO, v); else ptx::tmem_st16(tDO, v);
      }
      dpart[((u & 1u) * 2 + g) * BT + r] = part;
      ptx::mbar_arrive(dpart_full);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(stage_done);
      warp_arrive_leader(l_qd_ready);
      if (threadIdx.x == 64) {
        // every row thread of this CTA has read the six staging slots
        if (!ptx::mbar_wait(stage_done, u & 1u, w)) return false;
        for (int k = 0; k < 6; ++k) ptx::mbar_arrive(empty + slot(i0 + k));
      }
      return true;
    };
    auto next_unit = [&](int* rnd, int* bh, int* pq, int* split, int* j0, int* nk) {
      int b, bl;
      while (P.order.unit(pair, n_pairs, *rnd, &b, &bl)) {
        ++*rnd;
        if (dq_pair_unit<SPLIT>(P, bl, pq, split, j0, nk)) {
          *bh = b;
          return true;
        }
      }
      return false;
    };
    uint32_t item = 0, u_it = 0, sp = 0;
    int round = 0, bh, pq, split, j0, nk;
    bool have = next_unit(&round, &bh, &pq, &split, &j0, &nk);
    bool ok = !have || __all_sync(0xffffffffu, stage(0u, 0u));
    while (ok && have) {
      const int qt = 2 * pq + static_cast<int>(rank);
      const int q = qt * BT + r;
      const bool q_ok = q < Tq;
      const float lse = q_ok ? P.LSE[static_cast<size_t>(bh) * Tq + q] : -CUDART_INF_F;
      const float nlse2 = (lse == -CUDART_INF_F) ? -CUDART_INF_F : -lse * LOG2E;
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dpart_full, u_it & 1u, w)))) break;
      const float* dpu = dpart + (u_it & 1u) * 2 * BT;
      const float dd = dpu[r] + dpu[BT + r];
      // every row of the padded tile (the dK/dV kernel reads whole 128-row
      // slices); the second tile of the last pair may lie past the padding
      if (g == 0 && split == 0 && qt < P.n_q_tiles) {
        P.D[static_cast<size_t>(bh) * P.Tq_pad + q] = dd;
        P.NLSE2[static_cast<size_t>(bh) * P.Tq_pad + q] = nlse2;
      }
      for (int j = 0; j < nk; ++j, ++sp) {
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(s_full, sp & 1u, w)))) break;
        ptx::tc_fence_after();
        float p[64];
        {
          uint32_t v[2][32];
#pragma unroll
          for (int c = 0; c < 2; ++c) ptx::tmem_ld32(tS + c * 32, v[c]);
#pragma unroll
          for (int c = 0; c < 2; ++c) ptx::tmem_ld_wait(v[c]);
          ptx::tc_fence_before();
          warp_arrive_leader(l_s_free);
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 x = ptx::ffma2(make_float2(__uint_as_float(v[c][i]), __uint_as_float(v[c][i + 1])),
                                          make_float2(sc2, sc2), make_float2(nlse2, nlse2));
              p[c * 32 + i] = ptx::ex2(x.x);
              p[c * 32 + i + 1] = ptx::ex2(x.y);
            }
        }
        const int kv0 = (j0 + j) * BT + 64 * g;  // key of this thread's first column
        if (kv0 + 64 > Tk || (P.p.causal && kv0 + 63 > q)) {
          const int lim = min(Tk - kv0, P.p.causal ? q - kv0 + 1 : 64);   // columns [0, lim) allowed
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim) p[i] = 0.f;
        }
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dp_full, sp & 1u, w)))) break;
        ptx::tc_fence_after();
        uint32_t v[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) ptx::tmem_ld32(tDP + c * 32, v[c]);
#pragma unroll
        for (int c = 0; c < 2; ++c) ptx::tmem_ld_wait(v[c]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 e = ptx::fadd2(make_float2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1])),
                                        make_float2(-dd, -dd));
            const float2 rr = ptx::fmul2(make_float2(p[c * 32 + 2 * i], p[c * 32 + 2 * i + 1]), e);
            pk[i] = ptx::pack_bf16(rr.x, rr.y);
          }
          ptx::tmem_st16(tDP + c * 16, pk);   // over this group's own first 32 columns (already read)
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        warp_arrive_leader(l_ds_full);
      }
      if (!ok) break;
      const uint32_t i_next = item + 6 + 3 * nk;
      int nbh = 0, npq = 0, nsplit = 0, nj0 = 0, nnk = 0;
      const bool have_next = next_unit(&round, &nbh, &npq, &nsplit, &nj0, &nnk);
      if (have_next && !(ok = __all_sync(0xffffffffu, stage(i_next, u_it + 1)))) break;
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dq_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      if (SPLIT) {
        const size_t rows = static_cast<size_t>(P.p.B) * P.p.H * Tq;
        float* prow = P.dQpart + (static_cast<size_t>(split) * rows + static_cast<size_t>(bh) * Tq + (q_ok ? q : 0)) *
                                     C::HD + (C::HD / 2) * g;
#pragma unroll
        for (int c = 0; c < C::HD / 64; ++c) {
          uint32_t v[32];
          ptx::tmem_ld32(tDQ + c * 32, v);
          ptx::tmem_ld_wait(v);
          if (q_ok) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              reinterpret_cast<float4*>(prow + c * 32)[e] =
                  make_float4(__uint_as_float(v[4 * e]) * scale, __uint_as_float(v[4 * e + 1]) * scale,
                              __uint_as_float(v[4 * e + 2]) * scale, __uint_as_float(v[4 * e + 3]) * scale);
          }
        }
      } else {
        __nv_bfloat16* row = P.dQ + (static_cast<size_t>(bh) * Tq + (q_ok ? q : 0)) * C::HD + (C::HD / 2) * g;
#pragma unroll
        for (int c = 0; c < C::HD / 64; ++c) {
          uint32_t v[32];
          ptx::tmem_ld32(tDQ + c * 32, v);
          ptx::tmem_ld_wait(v);
          if (q_ok) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 a;
              a.x = ptx::pack_bf16(__uint_as_float(v[8 * e + 0]) * scale, __uint_as_float(v[8 * e + 1]) * scale);
              a.y = ptx::pack_bf16(__uint_as_float(v[8 * e + 2]) * scale, __uint_as_float(v[8 * e + 3]) * scale);
              a.z = ptx::pack_bf16(__uint_as_float(v[8 * e + 4]) * scale, __uint_as_float(v[8 * e + 5]) * scale);
              a.w = ptx::pack_bf16(__uint_as_float(v[8 * e + 6]) * scale, __uint_as_float(v[8 * e + 7]) * scale);
              reinterpret_cast<uint4*>(row + c * 32)[e] = a;
            }
          }
        }
      }
      // (the next unit's first dQ product, which overwrites the accumulator,
      // waits for both CTAs' first dS of that unit, written after this)
      ptx::tc_fence_before();
      item = i_next;
      ++u_it;
      have = have_next;
      bh = nbh;
      pq = npq;
      split = nsplit;
      j0 = nj0;
      nk = nnk;
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
template <int HV, bool SPLIT>
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
    cfg.blockDim = dim3(DQ_PAIR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = CfgP<HV>::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, dq_pair_kernel<HV, SPLIT>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    cached[dev] = n;
  }
  *out = cached[dev];
  return cudaSuccess;
}

template <int HV>
cudaError_t launch_dq_pair_t(const LaunchBwd& a, Params P) {
  using C = CfgP<HV>;
  const bool split = P.dq_splits > 1;
  const int n_pairs_q = (P.n_q_tiles + 1) / 2;
  const long long units = static_cast<long long>(n_pairs_q) * P.dq_splits * a.p.B * a.p.H;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  P.order = Order{n_pairs_q * P.dq_splits, a.p.B * a.p.H, a.p.causal ? 1 : 0};
  auto kern = split ? dq_pair_kernel<HV, true> : dq_pair_kernel<HV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int pairs = 0;
  e = split ? max_pairs<HV, true>(&pairs) : max_pairs<HV, false>(&pairs);
  if (e != cudaSuccess) return e;
  if (units < pairs) pairs = static_cast<int>(units);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(DQ_PAIR_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *a.tmQ64, *a.tmK64, *a.tmK, *a.tmV64, *a.tmdO64, *a.tmO64, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dq_pair(const LaunchBwd& a, const Params& P) {
  return a.p.dv == 128 ? launch_dq_pair_t<128>(a, P) : launch_dq_pair_t<64>(a, P);
}

}  // namespace bwd
}  // namespace attn
