// bf16 attention forward on tcgen05 tensor cores (sm_103a).
//
// Computes, per head, O = softmax(scale * Q K^T) V and LSE = log sum exp(scale
// * Q K^T) one 128-key tile at a time with an online softmax, never forming
// the Tq x Tk score matrix ("Tiled attention with an online softmax",
// section "Task"; "The Hidden Recurrence in Softmax Attention", section
// "Chunk-wise Mode with Online Softmax Re-scale"). Query tiles are the outer,
// parallel loop and key tiles the inner, sequential loop (the same page's
// "inner-outer loop exchange").
//
// One persistent CTA per SM walks a causal-aware list of work units. A unit is
// two 128-row query tiles (256 rows) of one head; both tiles share every K/V
// tile that TMA brings in. Warp roles (12 warps, 3 warpgroups):
//   warp 0      TMA producer (lane 0): Q, then K and V tiles through one ring
//   warp 1      MMA issuer (one elected lane); also allocates and frees TMEM
//   warps 2-3   idle (they complete the first warpgroup's register release)
//   warps 4-7   softmax group for query tile 0 (one thread per query row)
//   warps 8-11  softmax group for query tile 1
// The first warpgroup gives up registers (setmaxnreg) so each softmax thread
// can hold its whole 128-score row.
// TMEM (512 columns): tile t keeps its score tile S_t at columns [256t, 256t+128)
// and its accumulator O_t at [256t+128, 256t+128+dv). The softmax threads write
// P_t (bf16) over the first 64 columns of S_t, and the PV product reads it from
// there as the A operand. MMAs issued by one thread execute in order, so the
// next S_t product (which overwrites P_t) starts after the PV that reads it.
//
// Online softmax per query row, in log2 units s2 = s * scale * log2(e):
//   m_tile = max_j s2_j
//   if m_tile > m_used + TAU: rescale l and O by 2^(m_used - m_new), m_used = m_new
//   p_j = 2^(s2_j - m_used), l += sum p_j, O += P V
// Skipping the rescale while the running max grows by less than TAU keeps
// every p_j <= 2^TAU and leaves O/l and m_used + log2 l exact. A row with no
// allowed key yet uses 0 in place of m_used inside the exponentials (the
// page's -inf rule), so its p, l and O stay 0.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace fwd {

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per tile
constexpr int BOX_BYTES = 128 * 64 * 2;   // one TMA box: 128 rows x 64 bf16 (128-byte swizzle span)
constexpr float TAU = 8.0f;      // lazy-rescale threshold in log2 units
constexpr int NUM_THREADS = 384;   // three warpgroups
constexpr int REG_CTRL = 96;        // producer / MMA warpgroup
constexpr int REG_SOFTMAX = 200;   // each softmax warpgroup

// Tile widths HD >= d (Q and K rows) and HV >= dv (V and O rows), each 64 or
// 128; a narrower d or dv reads its missing columns as zeros through the
// tensor maps, and the epilogue writes only the first dv columns.
template <int HD, int HV>
struct Cfg {
  static constexpr int KB = HD / 64;                   // 64-column swizzle blocks per Q / K row
  static constexpr int KBV = HV / 64;                  // ... per V row
  static constexpr int TILE = BM * HD * 2;             // bytes of one 128-row Q or K tile
  static constexpr int TILE_V = BN * HV * 2;           // bytes of one 128-row V tile
  static constexpr int SLOT = TILE > TILE_V ? TILE : TILE_V;
  // K and V tiles share one FIFO ring of tile-sized slots, loaded in the
  // order they are consumed (K_0, V_0, K_1, V_1, ...). Five 32 KB slots give
  // every tile about two key steps of lead over its first use, which covers
  // the ~2 us a TMA load of a tile takes under load; the ring takes what the
  // two Q tiles leave of the shared memory, at most ten slots.
  static constexpr int NSLOT_FIT = (227 * 1024 - 2 * TILE - 1024) / SLOT;
  static constexpr int NSLOT = NSLOT_FIT < 10 ? NSLOT_FIT : 10;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + 2 * TILE;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * SLOT;
  // barriers: q_full, q_empty, full[NSLOT], empty[NSLOT], s_full[2], p_full[2], o_full[2], drain
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
  UnitOrder order;
  int n_kv_tiles;
  float sc2;   // scale * log2(e)
  // Split-KV mode (n_splits > 1): split s of a query-tile pair covers key
  // tiles [s * split_tiles, (s + 1) * split_tiles) and writes its normalised
  // partial output and log-sum-exp (fp32) to Opart [n_splits][B*H*Tq][dv]
  // and LSEpart [n_splits][B*H*Tq] instead of O and LSE.
  int n_splits;
  int split_tiles;
  float* Opart;
  float* LSEpart;
};

__device__ __forceinline__ void tile_counts(const Params& P, int qb, int* n0, int* n1) {
  const int nkb = P.n_kv_tiles;
  if (P.p.causal) {
    *n0 = min(2 * qb + 1, nkb);
    *n1 = min(2 * qb + 2, nkb);
  } else {
    *n0 = nkb;
    *n1 = nkb;
  }
}

// Key tiles of work unit `blk`: query-tile pair qb, first key tile j0, and
// n0 / n1 key tiles for its first / second query tile (n0 <= n1, possibly 0
// for the first tile of a split). False when the unit has no key tile.
template <bool SPLIT>
__device__ __forceinline__ bool unit_tiles(const Params& P, int blk, int* qb, int* j0, int* n0, int* n1) {
  if (!SPLIT) {
    *qb = blk;
    *j0 = 0;
    tile_counts(P, blk, n0, n1);
    return true;
  }
  *qb = blk / P.n_splits;
  const int s = blk - *qb * P.n_splits;
  int a0, a1;
  tile_counts(P, *qb, &a0, &a1);
  *j0 = s * P.split_tiles;
  *n0 = max(0, min(a0 - *j0, P.split_tiles));
  *n1 = max(0, min(a1 - *j0, P.split_tiles));
  return *n1 > 0;
}

// SPLIT: the split-KV variant (key ranges per unit, fp32 partial epilogue).
template <int HD, int HV, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params P) {
  using C = Cfg<HD, HV>;
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
  uint64_t* kv_full = bars + 2;            // [NSLOT]
  uint64_t* kv_empty = kv_full + C::NSLOT; // [NSLOT]
  uint64_t* s_full = kv_empty + C::NSLOT;  // [2]
  uint64_t* p_full = s_full + 2;        // [2]
  uint64_t* o_full = p_full + 2;        // [2]
  uint64_t* drain = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(kv_full + s, 1);
      ptx::mbar_init(kv_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(s_full + t, 1);
      ptx::mbar_init(p_full + t, 128);
      ptx::mbar_init(o_full + t, 1);
    }
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

  const int grid = gridDim.x;
  const int cta = blockIdx.x;

  const int wg = warp >> 2;
  if (wg == 0) {
   ptx::reg_release<REG_CTRL>();
   if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    // Item i of the K/V stream (i = 2 * tile + {0: K, 1: V}) goes to slot
    // i % NSLOT; the counters run across work units.
    ptx::WaitCtx w{abort_flag, P.status, 1u};
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
    uint32_t item = 0, u_it = 0, q_issued = 0;   // q_issued: Q loads issued (one per unit)
    bool ok = true;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &blk); ++round) {
      int qb, j0, n0, n1;
      if (!unit_tiles<SPLIT>(P, blk, &qb, &j0, &n0, &n1)) continue;
      if (!(ok = ptx::mbar_wait(q_empty, (u_it & 1u) ^ 1u, w))) break;
      ptx::mbar_arrive_expect_tx(q_full, 2 * C::TILE);
      for (int t = 0; t < 2; ++t)
        for (int b = 0; b < C::KB; ++b)
          ptx::tma_load_3d(sQ + t * C::TILE + b * BOX_BYTES, &tmQ, q_full, b * 64, (2 * qb + t) * BM, bh);
      q_issued = u_it + 1;
      for (int j = 0; ok && j < n1; ++j) {
        for (int kv = 0; kv < 2; ++kv, ++item) {
          const int sl = item % C::NSLOT;
          const uint32_t ph = (item / C::NSLOT) & 1u;
          if (!(ok = ptx::mbar_wait(kv_empty + sl, ph ^ 1u, w))) break;
          ptx::mbar_arrive_expect_tx(kv_full + sl, kv ? C::TILE_V : C::TILE);
          const CUtensorMap* map = kv ? &tmV : &tmK;
          for (int b = 0; b < (kv ? C::KBV : C::KB); ++b)
            ptx::tma_load_3d(sKV + sl * C::SLOT + b * BOX_BYTES, map, kv_full + sl, b * 64, (j0 + j) * BN, bh);
        }
      }
      ++u_it;
    }
    if (!ok) {
      // Let the copies already in flight land before the CTA exits.
      for (uint32_t n = (item > (uint32_t)C::NSLOT ? item - C::NSLOT : 0u); n < item; ++n)
        ptx::mbar_wait_drain(kv_full + n % C::NSLOT, (n / C::NSLOT) & 1u);
      // the last Q load issued (possibly this unit's, still in flight)
      if (q_issued > 0) ptx::mbar_wait_drain(q_full, (q_issued - 1) & 1u);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp follows the schedule and waits; the lane elect.sync
    // picks (lane 0) issues each step's MMAs and commits. A commit tracks the
    // MMAs of its own thread, so the issuing lane must not change; a change
    // is reported through the status word.
    ptx::WaitCtx w{abort_flag, P.status, 3u};
    const uint32_t sQa = ptx::smem_u32(sQ), sKVa = ptx::smem_u32(sKV);
    auto mma_S = [&](int t, int sl) {
      const uint32_t d = tmem + t * 256;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
        const uint64_t a = ptx::sdesc_advance(ptx::sdesc_sw128(sQa + t * C::TILE, 16, 1024), off);
        const uint64_t b = ptx::sdesc_advance(ptx::sdesc_sw128(sKVa + sl * C::SLOT, 16, 1024), off);
        ptx::mma_ss(d, a, b, C::IDESC_S, kk > 0 ? 1u : 0u);
      }
    };
    auto mma_PV = [&](int t, int sl, bool acc) {
      const uint32_t d = tmem + t * 256 + 128;
      const uint32_t a = tmem + t * 256;  // P_t, bf16 pairs in the first 64 columns of S_t
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t b = ptx::sdesc_advance(ptx::sdesc_sw128(sKVa + sl * C::SLOT, BOX_BYTES, 1024), kk * 2048);
        ptx::mma_ts(d, a + kk * 8, b, C::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
      }
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    // K_j is stream item 2 (kv_it + j), V_j item 2 (kv_it + j) + 1
    auto slot = [](uint32_t item) { return static_cast<int>(item % C::NSLOT); };
    auto par = [](uint32_t item) { return (item / C::NSLOT) & 1u; };
    uint32_t kv_it = 0, u_it = 0, pp[2] = {0u, 0u};
    bool ok = true, moved = false;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &blk); ++round) {
      int qb, j0, n0, n1;
      if (!unit_tiles<SPLIT>(P, blk, &qb, &j0, &n0, &n1)) continue;
      if (!(ok = wait(q_full, u_it & 1u))) break;
      const uint32_t ik = 2 * kv_it;
      if (!(ok = wait(kv_full + slot(ik), par(ik)))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        if (!SPLIT || n0 > 0) {   // (a split may hold no key tile for the first query tile)
          mma_S(0, slot(ik));
          ptx::mma_commit(s_full + 0);
        }
        mma_S(1, slot(ik));
        ptx::mma_commit(s_full + 1);
        ptx::mma_commit(kv_empty + slot(ik));
        if (n1 == 1) ptx::mma_commit(q_empty);   // no later MMA reads Q: the next unit's may load
      }
      __syncwarp();
      // V_0 and K_1: each step waits for the next step's tiles while its own
      // MMAs run, so only the softmax handshakes are left on the critical path
      if (!(ok = wait(kv_full + slot(ik + 1), par(ik + 1)))) break;
      if (n1 > 1 && !(ok = wait(kv_full + slot(ik + 2), par(ik + 2)))) break;
      for (int j = 0; j < n1; ++j) {
        const uint32_t iv = 2 * (kv_it + j) + 1, ikn = iv + 1;   // V_j, K_{j+1}: resident
        if (j < n0) {
          const bool more = j + 1 < n0;
          if (!(ok = wait(p_full + 0, pp[0] & 1u))) break;
          ++pp[0];
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_PV(0, slot(iv), j > 0);
            if (more) {
              mma_S(0, slot(ikn));
              ptx::mma_commit(s_full + 0);
            } else {
              ptx::mma_commit(o_full + 0);
            }
          }
          __syncwarp();
        }
        const bool more = j + 1 < n1;
        if (!(ok = wait(p_full + 1, pp[1] & 1u))) break;
        ++pp[1];
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
          mma_PV(1, slot(iv), j > 0);
          if (!more) ptx::mma_commit(o_full + 1);
          ptx::mma_commit(kv_empty + slot(iv));
          if (more) {
            mma_S(1, slot(ikn));
            ptx::mma_commit(s_full + 1);
            ptx::mma_commit(kv_empty + slot(ikn));
            // the unit's last S products are out (tile 0 ends no later than
            // tile 1): Q is free for the next unit during the last step
            if (j + 2 == n1) ptx::mma_commit(q_empty);
          }
        }
        __syncwarp();
        if (more && !(ok = wait(kv_full + slot(iv + 2), par(iv + 2)))) break;              // V_{j+1}
        if (j + 2 < n1 && !(ok = wait(kv_full + slot(ikn + 2), par(ikn + 2)))) break;   // K_{j+2}
      }
      if (!ok) break;
      kv_it += n1;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
   }
  } else {
    ptx::reg_acquire<REG_SOFTMAX>();
    // ------------------------------------------------------------ softmax
    const int t = wg - 1;                   // query tile of this group
    const int quad = warp & 3;              // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;         // row within the tile
    const uint32_t tS = tmem + (static_cast<uint32_t>(quad * 32) << 16) + t * 256;
    const uint32_t tO = tS + 128;
    ptx::WaitCtx w{abort_flag, P.status, 4u + t};
    const float sc2 = P.sc2;
    const int Tq = P.p.Tq, Tk = P.p.Tk;
    const int dv = P.p.dv;   // <= HV; a multiple of 8
    uint32_t sp = 0, op = 0;
    bool ok = true;
    int bh, blk;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &blk); ++round) {
      int qb, j0, n0, n1;
      if (!unit_tiles<SPLIT>(P, blk, &qb, &j0, &n0, &n1)) continue;
      const int nt = t ? n1 : n0;
      if (SPLIT && nt == 0) continue;   // nothing to write: the merge reads no partial for these rows
      const int qt = 2 * qb + t;
      const int q_row = qt * BM + r;
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        // every lane must agree before the warp-wide tcgen05 loads
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(s_full + t, sp & 1u, w)))) break;
        ++sp;
        ptx::tc_fence_after();
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, raw[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld_wait(raw[c]);
        float* s = reinterpret_cast<float*>(&raw[0][0]);
        const int kv0 = (j0 + j) * BN;
        const bool diag = P.p.causal && (kv0 + BN - 1 > qt * BM);
        if (diag || kv0 + BN > Tk) {
          const int lim = min(Tk - kv0, P.p.causal ? q_row - kv0 + 1 : BN);  // keys [0, lim) allowed
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) s[i] = -CUDART_INF_F;
        }
        // row max as 4 independent chains of three-input maxima
        float m4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmaxf(s[k], s[k + 4]);
#pragma unroll
        for (int i = 8; i < 128; i += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = ptx::fmax3(m4[k], s[i + k], s[i + 4 + k]);
        float mx = ptx::fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        mx *= sc2;
        const float m_new = fmaxf(m_used, mx);
        // Lazy rescale: move the reference max only when it grows by > TAU.
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
        // p = 2^(s * sc2 - ref), two lanes per fma / add instruction; the row
        // sum runs as 4 independent pairs of partial sums
        const float2 sc2v = make_float2(sc2, sc2), nrefv = make_float2(-ref, -ref);
        float2 ls[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ls[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 x = ptx::ffma2(make_float2(s[64 * h + 2 * i], s[64 * h + 2 * i + 1]), sc2v, nrefv);
            const float2 p = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            ls[i & 3] = ptx::fadd2(ls[i & 3], p);
            pk[i] = ptx::pack_bf16(p.x, p.y);
          }
          ptx::tmem_st32(tS + 32 * h, pk);
        }
        l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
        if (__any_sync(0xffffffffu, need)) {
          // O_t *= corr before the next PV product accumulates into it. The
          // previous PV into O_t is complete: it was issued before the S
          // product whose completion s_full reported.
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
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full + t);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(o_full + t, op & 1u, w)))) break;
      ++op;
      ptx::tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.0f / l : 0.f;
      const bool row_ok = q_row < Tq;
      const float lse_row = (l > 0.f) ? (m_used + log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
      if (SPLIT) {
        // partial result of this split: O_s = A / l in fp32 and LSE_s
        const size_t rows = static_cast<size_t>(P.p.B) * P.p.H * Tq;
        const size_t row = static_cast<size_t>(blk % P.n_splits) * rows + static_cast<size_t>(bh) * Tq +
                           (row_ok ? q_row : 0);
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
        continue;
      }
      __nv_bfloat16* orow = P.O + (static_cast<size_t>(bh) * Tq + (row_ok ? q_row : 0)) * dv;
#pragma unroll
      for (int c = 0; c < HV / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c * 32, o);
        ptx::tmem_ld_wait(o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (c * 32 + 8 * v < dv)   // dv < HV: the padded columns stay unwritten
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row_ok) P.LSE[static_cast<size_t>(bh) * Tq + q_row] = lse_row;
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int HD, int HV>
cudaError_t launch(const LaunchFwd& a) {
  using C = Cfg<HD, HV>;
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
  P.order.n_blocks = (a.p.Tq + 2 * BM - 1) / (2 * BM) * P.n_splits;
  P.order.n_heads = a.p.B * a.p.H;
  P.order.heavy_last = a.p.causal ? 1 : 0;
  P.sc2 = a.p.scale * 1.4426950408889634f;
  if (static_cast<long long>(P.order.n_blocks) * P.order.n_heads > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int units = P.order.count();
  const int grid = units < a.num_sms ? units : a.num_sms;
  auto kern = P.n_splits > 1 ? attn_fwd_bf16_kernel<HD, HV, true> : attn_fwd_bf16_kernel<HD, HV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // The register split must fit the launch allocation (see reg_acquire).
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs < REG_CTRL || fa.numRegs > REG_SOFTMAX || 3 * fa.numRegs < REG_CTRL + 2 * REG_SOFTMAX)
    return cudaErrorInvalidConfiguration;
  kern<<<grid, NUM_THREADS, C::SMEM, a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, P);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd_bf16(const LaunchFwd& a) {
  // d or dv below the tile width runs on the next width up (zero columns)
  if (a.p.d > 64) return a.p.dv > 64 ? fwd::launch<128, 128>(a) : fwd::launch<128, 64>(a);
  return a.p.dv > 64 ? fwd::launch<64, 128>(a) : fwd::launch<64, 64>(a);
}

}  // namespace attn
