// bf16 attention backward on tcgen05 tensor cores (sm_103a).
//
// Recomputes P tile by tile from the stored log-sum-exp instead of keeping
// it ("The Hidden Recurrence in Softmax Attention", section "Flash Attention
// Backward Pass"), and forms the gradient terms of "attention_backprop"
// (sections "Gradient of V and P", "Gradient of S", "Gradient of Q and K"):
//   D  = rowsum(dO o O)                        (dQ kernel, or the preprocess kernel in atomic mode)
//   P  = exp(scale * Q K^T - LSE)
//   dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D)
//   dK = scale * dS^T Q,          dQ = scale * dS K
//
// dK/dV kernel: one persistent CTA per SM; a work unit is one 128-key tile of
// one head, and the CTA loops over the query tiles that can see it. K and V
// stay in shared memory for the whole unit; Q, dO (TMA) and the 128-row slices
// of NLSE2 and D (bulk copies) stream through rings of their own. Warp roles
// (16 warps, 4 warpgroups):
//   warp 0       producer (lane 0 issues the TMA and bulk copies)
//   warp 1       MMA issuer (lane 0); allocates and frees TMEM
//   warps 2-3    idle (they complete the first warpgroup's register release)
//   warps 4-7    P / dS, query columns 0-63 of the tile (one thread per key row)
//   warps 8-11   P / dS, query columns 64-127
//   warps 12-15  dQ group: reads each dQ tile out of TMEM, stages it in the dS
//                buffer in two 64-column halves and adds it into the fp32
//                accumulator with TMA reduce-add; writes dK and dV per unit
// setmaxnreg splits the launch's 512 x 128 registers as 104 / 152 / 152 / 104
// (atomic dQ) or 96 / 168 / 168 / 80 (deterministic).
// TMEM (512 columns): dV [0,128), dK [128,256), S^T [256,384), dP^T [384,512).
// Per query tile the MMA warp issues
//   S^T  = K Q^T        (A = K, B = Q, both K-major in smem)
//   dP^T = V dO^T       (A = V, B = dO)
//   dV  += P^T dO       (A = P^T bf16 in TMEM over S^T, B = dO MN-major)
//   dK  += dS^T Q       (A = dS^T bf16 in TMEM over dP^T, B = Q MN-major)
//   dQ   = dS K         (A = dS from smem, MN-major; B = K MN-major) -> over dP^T
// The last product is skipped in deterministic mode, where a separate dQ
// kernel (a unit per query tile looping over key tiles in a fixed order, or
// per query tile and key range when query tiles are few) accumulates dQ in
// TMEM and writes it once (or its range's fp32 partial, added in order by
// reduce_dq_kernel). That kernel keeps Q and dO in TMEM as the A operands of
// S = Q K^T and dP = dO V^T, so all three of its products per key tile read
// only a K or V tile from shared memory. The dQ and dK/dV kernels take d (Q, K, dQ, dK) and dv (V,
// O, dO, dV) as separate template parameters, each 64 or 128.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "bwd_common.cuh"
#include "ptx.cuh"

namespace attn {
namespace bwd {

constexpr int KV_THREADS = 512;          // dK/dV kernel: four warpgroups
// Per-warpgroup register budgets of the dK/dV kernel (setmaxnreg). The
// deterministic variant has no dQ staging in its last warpgroup (only the
// dK/dV epilogue) and gives the P/dS threads room to hold a tile's 64
// LSE and D values in registers.
template <bool ATOMIC_DQ>
struct KvRegs {
  static constexpr int CTRL = ATOMIC_DQ ? 104 : 96;   // producer / MMA warpgroup
  static constexpr int PDS = ATOMIC_DQ ? 152 : 168;   // each of the two P / dS warpgroups
  static constexpr int DQ = ATOMIC_DQ ? 104 : 80;     // dQ / epilogue warpgroup
};
constexpr int KV_REG_LAUNCH = 128;       // 65536 / 512, what the launch bound gives

// Query tiles [first, first + count) that see key tile kb.
__device__ __forceinline__ void q_range(const Params& P, int kb, int* first, int* count) {
  const int f = P.p.causal ? kb : 0;
  *first = f;
  *count = P.n_q_tiles > f ? P.n_q_tiles - f : 0;
}

// HD = d (Q, K, dQ, dK rows), HV = dv (V, O, dO, dV rows); each 64 or 128.
template <int HD, int HV, bool ATOMIC_DQ>
struct CfgKV {
  static constexpr int KB = HD / 64;        // 64-column boxes per Q / K row
  static constexpr int KBV = HV / 64;       // ... per V / dO row
  static constexpr int TILE = BT * HD * 2;  // one 128-row Q or K tile
  static constexpr int TILE_V = BT * HV * 2;  // one 128-row V or dO tile
  // Q tiles, dO tiles and the -LSE*log2(e) / D slices of a query tile have
  // rings of their own. A Q tile stays resident from its S^T product to its
  // dK product at the end of the step, a dO tile from its dP^T product to its
  // dV product in the middle of the next one, the slices until the P/dS
  // threads finish the step. The deterministic variant, which needs no dS
  // buffer in shared memory, gives Q three slots; atomic mode keeps two.
  static constexpr int NQ = ATOMIC_DQ ? 2 : 3;
  static constexpr int NO = 2;
  static constexpr int NL = 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE_V;        // [NQ]
  static constexpr int OFF_DO = OFF_Q + NQ * TILE;    // [NO]
  // atomic mode: dS, 128 q x 128 keys bf16, MN-major; it then stages one
  // 64-column half of the fp32 dQ tile (two 128 x 32 boxes) for the TMA reduce
  static constexpr int OFF_DS = OFF_DO + NO * TILE_V;
  static constexpr int DS_BYTES = ATOMIC_DQ ? BT * BT * 2 : 0;
  static constexpr int OFF_LSE = OFF_DS + DS_BYTES;   // [NL][128] fp32 (-LSE * log2 e, -inf = no key)
  static constexpr int OFF_D = OFF_LSE + NL * BT * 4; // [NL][128] fp32
  static constexpr int OFF_BAR = OFF_D + NL * BT * 4;
  // kv_full, kv_empty, q_full[NQ], q_empty[NQ], o_full[NO], o_empty[NO], l_full[NL], l_empty[NL],
  // s_full, dp_full, p_full, ds_full, dq_full, dq_free, acc_full, dv_free, stage_full, stage_free,
  // sds_free, drain, dk_free
  // ..., unit queue full[4], empty[4]
  static constexpr int NBAR = 2 + 2 * NQ + 2 * NO + 2 * NL + 13 + 2 * UnitQueue::N;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM address, abort word, unit queue slots
  static constexpr int SMEM = OFF_MISC + 16 + 4 * UnitQueue::N;
  static constexpr int UQ_READERS = 1 + 256 + 128;   // the MMA warp (once), every P/dS and epilogue thread
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16(BT, BT, false, false);
  static constexpr uint32_t IDESC_DV = ptx::idesc_bf16(BT, HV, false, true);    // dV (A in TMEM)
  static constexpr uint32_t IDESC_DK = ptx::idesc_bf16(BT, HD, false, true);    // dK (A in TMEM)
  static constexpr uint32_t IDESC_DQ = ptx::idesc_bf16(BT, HD, true, true);     // dQ = dS K
};


// DYN: units claimed at run time through the unit queue (see UnitQueue);
// otherwise the static order, with no queue code compiled in.
template <int HD, int HV, bool ATOMIC_DQ, bool DYN>
__global__ void __launch_bounds__(KV_THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdQ, const Params P) {
  using C = CfgKV<HD, HV, ATOMIC_DQ>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sdO = smem + C::OFF_DO;
  uint8_t* sdS = smem + C::OFF_DS;
  float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* sD = reinterpret_cast<float*>(smem + C::OFF_D);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;             // [NQ]
  uint64_t* q_empty = q_full + C::NQ;      // [NQ]
  uint64_t* o_full = q_empty + C::NQ;      // [NO]
  uint64_t* o_empty = o_full + C::NO;      // [NO]
  uint64_t* l_full = o_empty + C::NO;      // [NL]
  uint64_t* l_empty = l_full + C::NL;      // [NL]
  uint64_t* s_full = l_empty + C::NL;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* ds_full = s_full + 3;
  uint64_t* dq_full = s_full + 4;
  uint64_t* dq_free = s_full + 5;
  uint64_t* acc_full = s_full + 6;
  uint64_t* dv_free = s_full + 7;    // the epilogue has read the dV accumulator
  uint64_t* dk_free = s_full + 12;   // ... and the dK accumulator
  uint64_t* stage_full = s_full + 8;
  uint64_t* stage_free = s_full + 9;
  uint64_t* sds_free = s_full + 10;
  uint64_t* drain = s_full + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  const UnitQueue uq{reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16), s_full + 13,
                     s_full + 13 + UnitQueue::N};

  if (threadIdx.x == 0) {
    for (int s = 0; s < UnitQueue::N; ++s) {
      ptx::mbar_init(uq.full + s, 1);
      ptx::mbar_init(uq.empty + s, C::UQ_READERS);
    }
    ptx::mbar_init(kv_full, 1);
    ptx::mbar_init(kv_empty, 1);
    for (int s = 0; s < C::NQ; ++s) {
      ptx::mbar_init(q_full + s, 1);
      ptx::mbar_init(q_empty + s, 1);
    }
    for (int s = 0; s < C::NO; ++s) {
      ptx::mbar_init(o_full + s, 1);
      ptx::mbar_init(o_empty + s, 1);
    }
    for (int s = 0; s < C::NL; ++s) {
      ptx::mbar_init(l_full + s, 1);
      ptx::mbar_init(l_empty + s, 256);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(p_full, 256);
    ptx::mbar_init(ds_full, 256);
    ptx::mbar_init(dq_full, 1);
    ptx::mbar_init(dq_free, 128);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(dv_free, 128);
    ptx::mbar_init(dk_free, 128);
    ptx::mbar_init(stage_full, 128);
    ptx::mbar_init(stage_free, 1);
    ptx::mbar_init(sds_free, 1);
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
  const uint32_t T_DV = 0, T_DK = 128, T_ST = 256, T_DP = 384;
  // Query tile number n (counted across units) uses Q slot n % NQ and dO slot n % NO.
  auto qslot = [](uint32_t n) { return static_cast<int>(n % C::NQ); };
  auto qpar = [](uint32_t n) { return (n / C::NQ) & 1u; };
  auto oslot = [](uint32_t n) { return static_cast<int>(n % C::NO); };
  auto opar = [](uint32_t n) { return (n / C::NO) & 1u; };
  auto lslot = [](uint32_t n) { return static_cast<int>(n % C::NL); };
  auto lpar = [](uint32_t n) { return (n / C::NL) & 1u; };

  const int Tk = P.p.Tk;
  const int wg = warp >> 2;
  // the launch's units: 128-key tiles of every head, handed out at run time
  // in head groups, the longest (causal: first) key tiles first
  const int nb = P.n_k_tiles, nh = P.p.B * P.p.H, total = nb * nh;
  const int cta = blockIdx.x, grid = gridDim.x;
  auto decode = [&](int x, int* bh, int* kb) { grouped_unit(x, nb, nh, P.group, false, bh, kb); };

  if (wg == 0) {
    ptx::reg_release<KvRegs<ATOMIC_DQ>::CTRL>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      ptx::WaitCtx w{abort_flag, P.status, 1u};
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      ptx::tma_prefetch_desc(&tmdO);
      uint32_t u_it = 0, q_it = 0, q_issued = 0, o_issued = 0, l_issued = 0, pu = 0;
      int bh = 0, kb = 0;
      // take the next unit and publish it (the one after it before this
      // one's tiles load)
      int x = DYN ? next_unit_index(P, pu, cta, grid, total) : 0;
      bool ok = true;
      if constexpr (DYN) ok = uq_push(uq, pu, x, w);
      ++pu;
      while (ok && x < total) {
        if constexpr (DYN) {
          const int xn = next_unit_index(P, pu, cta, grid, total);
          if (!(ok = uq_push(uq, pu, xn, w))) break;
          decode(x, &bh, &kb);
          x = xn;
        } else if (!P.order.unit(cta, grid, static_cast<int>(pu) - 1, &bh, &kb)) {
          break;
        }
        ++pu;
        int q0, nq;
        q_range(P, kb, &q0, &nq);
        if (nq == 0) continue;
        if (!(ok = ptx::mbar_wait(kv_empty, (u_it & 1u) ^ 1u, w))) break;
        ptx::mbar_arrive_expect_tx(kv_full, C::TILE + C::TILE_V);
        for (int b = 0; b < C::KB; ++b) ptx::tma_load_3d(sK + b * BOX_BYTES, &tmK, kv_full, b * 64, kb * BT, bh);
        for (int b = 0; b < C::KBV; ++b) ptx::tma_load_3d(sV + b * BOX_BYTES, &tmV, kv_full, b * 64, kb * BT, bh);
        for (int ii = 0; ii < nq; ++ii, ++q_it) {
          const int qs = qslot(q_it), os = oslot(q_it);
          const int qt = q0 + ii;
          const size_t row0 = static_cast<size_t>(bh) * P.Tq_pad + static_cast<size_t>(qt) * BT;
          if (!(ok = ptx::mbar_wait(q_empty + qs, qpar(q_it) ^ 1u, w))) break;
          ptx::mbar_arrive_expect_tx(q_full + qs, C::TILE);
          for (int b = 0; b < C::KB; ++b)
            ptx::tma_load_3d(sQ + qs * C::TILE + b * BOX_BYTES, &tmQ, q_full + qs, b * 64, qt * BT, bh);
          q_issued = q_it + 1;
          const int ls = lslot(q_it);
          if (!(ok = ptx::mbar_wait(l_empty + ls, lpar(q_it) ^ 1u, w))) break;
          ptx::mbar_arrive_expect_tx(l_full + ls, 2 * BT * 4);
          ptx::bulk_load(sLSE + ls * BT, P.NLSE2 + row0, BT * 4, l_full + ls);
          ptx::bulk_load(sD + ls * BT, P.D + row0, BT * 4, l_full + ls);
          l_issued = q_it + 1;
          if (!(ok = ptx::mbar_wait(o_empty + os, opar(q_it) ^ 1u, w))) break;
          ptx::mbar_arrive_expect_tx(o_full + os, C::TILE_V);
          for (int b = 0; b < C::KBV; ++b)
            ptx::tma_load_3d(sdO + os * C::TILE_V + b * BOX_BYTES, &tmdO, o_full + os, b * 64, qt * BT, bh);
          o_issued = q_it + 1;
        }
        ++u_it;
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        if (u_it > 0 || q_it > 0) ptx::mbar_wait_drain(kv_full, u_it & 1u);
        for (uint32_t n = (q_issued > (uint32_t)C::NQ ? q_issued - C::NQ : 0u); n < q_issued; ++n)
          ptx::mbar_wait_drain(q_full + qslot(n), qpar(n));
        for (uint32_t n = (o_issued > (uint32_t)C::NO ? o_issued - C::NO : 0u); n < o_issued; ++n)
          ptx::mbar_wait_drain(o_full + oslot(n), opar(n));
        for (uint32_t n = (l_issued > (uint32_t)C::NL ? l_issued - C::NL : 0u); n < l_issued; ++n)
          ptx::mbar_wait_drain(l_full + lslot(n), lpar(n));
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp follows the schedule and waits; the lane elect.sync
      // picks (lane 0) issues the MMAs and commits. A commit tracks the MMAs
      // of its own thread, so the issuing lane must not change; a change is
      // reported through the status word.
      ptx::WaitCtx w{abort_flag, P.status, 2u};
      const uint32_t aK = ptx::smem_u32(sK), aV = ptx::smem_u32(sV), aQ = ptx::smem_u32(sQ),
                     adO = ptx::smem_u32(sdO), adS = ptx::smem_u32(sdS);
      auto kmaj = [](uint32_t base, int kk) {  // K-major operand, k-step kk of 16 elements
        return ptx::sdesc_advance(ptx::sdesc_sw128(base, 16, 1024), (kk >> 2) * BOX_BYTES + (kk & 3) * 32);
      };
      auto mnmaj = [](uint32_t base, int kk) {  // MN-major operand, k-step kk of 16 rows
        return ptx::sdesc_advance(ptx::sdesc_sw128(base, BOX_BYTES, 1024), kk * 2048);
      };
      auto mma_st = [&](uint32_t n) {   // S^T = K Q^T for query tile n
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_ss(tmem + T_ST, kmaj(aK, kk), kmaj(aQ + qslot(n) * C::TILE, kk), C::IDESC_S, kk > 0);
      };
      auto mma_dpt = [&](uint32_t n) {   // dP^T = V dO^T for query tile n
#pragma unroll
        for (int kk = 0; kk < HV / 16; ++kk)
          ptx::mma_ss(tmem + T_DP, kmaj(aV, kk), kmaj(adO + oslot(n) * C::TILE_V, kk), C::IDESC_S, kk > 0);
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
      };
      uint32_t u_it = 0, q_it = 0, pp = 0, dqf = 0, ru = 0;
      bool ok = true, moved = false;
      int bh, kb;
      while (ok) {
        if constexpr (DYN) {
          int x;
          if (!(ok = uq_read(uq, ru, &x, w))) break;
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(uq.empty + ru % UnitQueue::N);
          if (x >= total) break;
          decode(x, &bh, &kb);
        } else if (!P.order.unit(cta, grid, static_cast<int>(ru), &bh, &kb)) {
          break;
        }
        ++ru;
        int q0, nq;
        q_range(P, kb, &q0, &nq);
        if (nq == 0) continue;
        if (!(ok = wait(kv_full, u_it & 1u))) break;
        {
          if (!(ok = wait(q_full + qslot(q_it), qpar(q_it)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_st(q_it);
            ptx::mma_commit(s_full);
          }
          __syncwarp();
          if (ATOMIC_DQ && dqf > 0) {
            if (!(ok = wait(dq_free, (dqf - 1) & 1u))) break;
          }
          if (!(ok = wait(o_full + oslot(q_it), opar(q_it)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_dpt(q_it);
            ptx::mma_commit(dp_full);
            // deterministic: K and V are read by no later MMA of a one-tile
            // unit, so the next unit's tiles may start loading now
            if (!ATOMIC_DQ && nq == 1) ptx::mma_commit(kv_empty);
          }
          __syncwarp();
          // Q and dO of the next query tile: each step waits for the tiles of
          // the step after it while its own MMAs run, so only the P/dS
          // handshakes are left on the critical path
          if (nq > 1 && !(ok = wait(q_full + qslot(q_it + 1), qpar(q_it + 1)))) break;
        }
        for (int ii = 0; ii < nq; ++ii) {
          const uint32_t it = q_it + ii;
          const bool more = ii + 1 < nq;   // Q of tile it + 1 is resident
          // dV += P^T dO, then the next S^T (it overwrites P^T only after the
          // product above has read it). The first dV (dK) of a unit
          // overwrites the accumulator: the epilogue must have read the
          // previous unit's (its S^T and dP^T products overlap that epilogue).
          if (ii == 0 && !(ok = wait(dv_free, (u_it & 1u) ^ 1u))) break;
          if (!(ok = wait(p_full, pp & 1u))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              ptx::mma_ts(tmem + T_DV, tmem + T_ST + packed_col(kk), mnmaj(adO + oslot(it) * C::TILE_V, kk),
                          C::IDESC_DV, (ii > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(o_empty + oslot(it));
            if (more) {
              mma_st(it + 1);
              ptx::mma_commit(s_full);
            }
          }
          __syncwarp();
          // dK += dS^T Q (and, atomic mode, dQ = dS K into the dP^T columns)
          if (ii == 0 && !(ok = wait(dk_free, (u_it & 1u) ^ 1u))) break;
          if (!(ok = wait(ds_full, pp & 1u))) break;
          ++pp;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              ptx::mma_ts(tmem + T_DK, tmem + T_DP + packed_col(kk), mnmaj(aQ + qslot(it) * C::TILE, kk),
                          C::IDESC_DK, (ii > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(q_empty + qslot(it));
            if (ATOMIC_DQ) {
#pragma unroll
              for (int kk = 0; kk < BT / 16; ++kk)
                ptx::mma_ss(tmem + T_DP, mnmaj(adS, kk), mnmaj(aK, kk), C::IDESC_DQ, kk > 0);
              ptx::mma_commit(dq_full);
            }
          }
          __syncwarp();
          if (ATOMIC_DQ) ++dqf;
          if (more) {
            if (ATOMIC_DQ) {
              if (!(ok = wait(dq_free, (dqf - 1) & 1u))) break;
            }
            if (!(ok = wait(o_full + oslot(it + 1), opar(it + 1)))) break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
              moved |= lane != 0;
              mma_dpt(it + 1);
              ptx::mma_commit(dp_full);
              // deterministic: that was the last MMA reading K or V in this
              // unit (the last S^T went out with dV above), so the next
              // unit's K and V may start loading during the last step
              if (!ATOMIC_DQ && ii + 2 == nq) ptx::mma_commit(kv_empty);
            }
            __syncwarp();
          }
          if (ii + 2 < nq && !(ok = wait(q_full + qslot(it + 2), qpar(it + 2)))) break;
        }
        if (!ok) break;
        if (ptx::elect_one()) {
          moved |= lane != 0;
          ptx::mma_commit(acc_full);
          if (ATOMIC_DQ) ptx::mma_commit(kv_empty);   // the dQ products read K up to the last step
        }
        __syncwarp();
        q_it += nq;
        ++u_it;
      }
      if (!ok) {
        if (ptx::elect_one()) ptx::mma_commit(drain);
        __syncwarp();
        ptx::mbar_wait_drain(drain, 0u);
      }
      if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
    }
  } else if (wg <= 2) {
    ptx::reg_acquire<KvRegs<ATOMIC_DQ>::PDS>();
    // ------------------------------------------------------------ P / dS (thread = key row)
    // Group h handles query columns [64h, 64h + 64) of the tile.
    const int h = wg - 1;
    const int quad = warp & 3;
    const int j = quad * 32 + lane;                 // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tST = tmem + lane_off + T_ST + 64 * h, tDP = tmem + lane_off + T_DP + 64 * h;
    ptx::WaitCtx w{abort_flag, P.status, 3u};
    const float sc2 = P.sc2;
    const float2 sc2v = make_float2(sc2, sc2), neg1 = make_float2(-1.f, -1.f);
    uint32_t q_it = 0, sp = 0, ru = 0;
    bool ok = true;
    int bh, kb;
    while (ok) {
      if constexpr (DYN) {
        int x;
        if (!(ok = uq_read(uq, ru, &x, w))) break;
        ptx::mbar_arrive(uq.empty + ru % UnitQueue::N);
        if (x >= total) break;
        decode(x, &bh, &kb);
      } else if (!P.order.unit(cta, grid, static_cast<int>(ru), &bh, &kb)) {
        break;
      }
      ++ru;
      int q0, nq;
      q_range(P, kb, &q0, &nq);
      if (nq == 0) continue;
      const int key = kb * BT + j;
      const bool key_ok = key < Tk;
      for (int ii = 0; ii < nq; ++ii, ++q_it, ++sp) {
        const int ls = lslot(q_it);
        const int qt = q0 + ii;
        const float* nlse2 = sLSE + ls * BT + 64 * h;
        const float* dd = sD + ls * BT + 64 * h;
        // the staged LSE / D slices of this tile are visible once l_full completed
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(l_full + ls, lpar(q_it), w)))) break;
        // deterministic: this tile's 64 -LSE*log2(e) values into registers
        // while S^T is being computed
        float nl[ATOMIC_DQ ? 1 : 64];
        if (!ATOMIC_DQ) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 t4 = reinterpret_cast<const float4*>(nlse2)[i];
            nl[4 * i] = t4.x;
            nl[4 * i + 1] = t4.y;
            nl[4 * i + 2] = t4.z;
            nl[4 * i + 3] = t4.w;
          }
        }
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(s_full, sp & 1u, w)))) break;
        ptx::tc_fence_after();
        // pass 1: P^T_j,q = 2^(s * scale * log2e - LSE_q * log2e), masked; packed bf16
        // over the first half of this group's S^T columns. The packed values
        // stay in registers for pass 2: once p_full is signalled the MMA warp
        // may overwrite S^T with the next tile's scores.
        uint32_t pkeep[2][16];
        {
          uint32_t rs[2][32];
          ptx::tmem_ld32(tST, rs[0]);
          ptx::tmem_ld32(tST + 32, rs[1]);
          ptx::tmem_ld_wait(rs[0]);
          ptx::tmem_ld_wait(rs[1]);
          // query column (within this group) below which P = 0: the diagonal
          // tile of the causal mask, or every column for a key past Tk
          const int lim = !key_ok ? 64 : (P.p.causal && qt == kb ? j - 64 * h : 0);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const int qa = c * 32 + 2 * i;
              const float4 l4 = ATOMIC_DQ ? ptx::lds128(nlse2 + qa)
                                          : make_float4(nl[qa & 63], nl[(qa + 1) & 63], nl[(qa + 2) & 63],
                                                        nl[(qa + 3) & 63]);
              const float2 x01 = ptx::ffma2(make_float2(__uint_as_float(rs[c][2 * i]), __uint_as_float(rs[c][2 * i + 1])),
                                            sc2v, make_float2(l4.x, l4.y));
              const float2 x23 = ptx::ffma2(make_float2(__uint_as_float(rs[c][2 * i + 2]),
                                                        __uint_as_float(rs[c][2 * i + 3])),
                                            sc2v, make_float2(l4.z, l4.w));
              float p0 = ptx::ex2(x01.x), p1 = ptx::ex2(x01.y), p2 = ptx::ex2(x23.x), p3 = ptx::ex2(x23.y);
              if (lim > 0) {
                if (qa < lim) p0 = 0.f;
                if (qa + 1 < lim) p1 = 0.f;
                if (qa + 2 < lim) p2 = 0.f;
                if (qa + 3 < lim) p3 = 0.f;
              }
              pkeep[c][i] = ptx::pack_bf16(p0, p1);
              pkeep[c][i + 1] = ptx::pack_bf16(p2, p3);
            }
            ptx::tmem_st16(tST + c * 16, pkeep[c]);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full);
        // pass 2: dS^T_j,q = P^T (dP^T - D_q); bf16 over dP^T and into smem (dS, MN-major)
        float dl[ATOMIC_DQ ? 1 : 64];
        if (!ATOMIC_DQ) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 t4 = reinterpret_cast<const float4*>(dd)[i];
            dl[4 * i] = t4.x;
            dl[4 * i + 1] = t4.y;
            dl[4 * i + 2] = t4.z;
            dl[4 * i + 3] = t4.w;
          }
        }
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dp_full, sp & 1u, w)))) break;
        if (ATOMIC_DQ) {
          // the dQ group has finished staging the previous dQ tile in the dS buffer
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(sds_free, (q_it & 1u) ^ 1u, w)))) break;
        }
        ptx::tc_fence_after();
        {
          uint32_t rd[2][32];
          ptx::tmem_ld32(tDP, rd[0]);
          ptx::tmem_ld32(tDP + 32, rd[1]);
          ptx::tmem_ld_wait(rd[0]);
          ptx::tmem_ld_wait(rd[1]);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const int qa = c * 32 + 2 * i;
              const float4 d4 = ATOMIC_DQ ? ptx::lds128(dd + qa)
                                          : make_float4(dl[qa & 63], dl[(qa + 1) & 63], dl[(qa + 2) & 63],
                                                        dl[(qa + 3) & 63]);
              const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pkeep[c][i]));
              const float2 pg = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pkeep[c][i + 1]));
              // (dP - D) as -D * 1 + dP, two lanes per instruction
              const float2 e01 = ptx::ffma2(make_float2(d4.x, d4.y), neg1,
                                            make_float2(__uint_as_float(rd[c][2 * i]), __uint_as_float(rd[c][2 * i + 1])));
              const float2 e23 = ptx::ffma2(make_float2(d4.z, d4.w), neg1,
                                            make_float2(__uint_as_float(rd[c][2 * i + 2]),
                                                        __uint_as_float(rd[c][2 * i + 3])));
              const float2 s01 = ptx::fmul2(pf, e01), s23 = ptx::fmul2(pg, e23);
              pk[i] = ptx::pack_bf16(s01.x, s01.y);
              pk[i + 1] = ptx::pack_bf16(s23.x, s23.y);
            }
            ptx::tmem_st16(tDP + c * 16, pk);
            if (ATOMIC_DQ) {
              // dS is MN-major for the dQ product: row = key j, column = query
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint32_t off = sw128_offset(j, 64 * h + c * 32 + v * 8);
                *reinterpret_cast<uint4*>(sdS + off) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              }
            }
          }
        }
        ptx::tmem_st_wait();
        if (ATOMIC_DQ) ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ds_full);
        ptx::mbar_arrive(l_empty + ls);   // done with this tile's LSE / D slices
      }
    }
  } else {
    ptx::reg_release<KvRegs<ATOMIC_DQ>::DQ>();
    // ------------------------------------------------------------ dQ reduce; dK / dV epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                 // TMEM lane = row
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool leader = (threadIdx.x == 3 * 128);
    ptx::WaitCtx w{abort_flag, P.status, 4u};
    const float scale = P.p.scale;
    uint32_t u_it = 0, dqf = 0, sfull = 0;
    bool ok = true;
    int bh, kb;
    // one 64-column half of the fp32 dQ tile into the staging boxes (128-byte
    // swizzle: 16-byte chunk c of row r at chunk position c ^ (r & 7))
    auto stage_half = [&](const uint32_t (&v)[2][32]) {
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 x = make_uint4(__float_as_uint(__uint_as_float(v[b][4 * c]) * scale),
                               __float_as_uint(__uint_as_float(v[b][4 * c + 1]) * scale),
                               __float_as_uint(__uint_as_float(v[b][4 * c + 2]) * scale),
                               __float_as_uint(__uint_as_float(v[b][4 * c + 3]) * scale));
          *reinterpret_cast<uint4*>(sdS + b * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = x;
        }
    };
    uint32_t ru = 0;
    while (ok) {
      if constexpr (DYN) {
        int x;
        if (!(ok = uq_read(uq, ru, &x, w))) break;
        ptx::mbar_arrive(uq.empty + ru % UnitQueue::N);
        if (x >= total) break;
        decode(x, &bh, &kb);
      } else if (!P.order.unit(cta, grid, static_cast<int>(ru), &bh, &kb)) {
        break;
      }
      ++ru;
      int q0, nq;
      q_range(P, kb, &q0, &nq);
      const int key = kb * BT + r;
      const bool key_ok = key < Tk;
      __nv_bfloat16* dk_row = P.dK + (static_cast<size_t>(bh) * Tk + (key_ok ? key : 0)) * HD;
      __nv_bfloat16* dv_row = P.dV + (static_cast<size_t>(bh) * Tk + (key_ok ? key : 0)) * HV;
      if (nq == 0) {
        if (key_ok) {
          for (int c = 0; c < HD / 8; ++c) reinterpret_cast<uint4*>(dk_row)[c] = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < HV / 8; ++c) reinterpret_cast<uint4*>(dv_row)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      if (ATOMIC_DQ) {
        for (int ii = 0; ii < nq; ++ii, ++dqf) {
          const int qt = q0 + ii;
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dq_full, dqf & 1u, w)))) break;
          ptx::tc_fence_after();
          for (int half = 0; half < HD / 64; ++half) {
            uint32_t v[2][32];
            ptx::tmem_ld32(tmem + lane_off + T_DP + 64 * half, v[0]);
            ptx::tmem_ld32(tmem + lane_off + T_DP + 64 * half + 32, v[1]);
            ptx::tmem_ld_wait(v[0]);
            ptx::tmem_ld_wait(v[1]);
            if (half == HD / 64 - 1) {
              // the whole tile is in registers: hand the TMEM columns back
              ptx::tc_fence_before();
              ptx::mbar_arrive(dq_free);
            }
            if (half > 0) {
              // the copy engine has read the previous half out of the buffer
              if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(stage_free, (dqf & 1u), w)))) break;
            }
            stage_half(v);
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(stage_full);
            if (leader) {
              if (ptx::mbar_wait(stage_full, sfull & 1u, w)) {
                ptx::tma_reduce_add_3d(&tmdQ, sdS, 64 * half, qt * BT, bh);
                ptx::tma_reduce_add_3d(&tmdQ, sdS + 16384, 64 * half + 32, qt * BT, bh);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read0();
                ptx::mbar_arrive(half == HD / 64 - 1 ? sds_free : stage_free);
              } else {
                ok = false;
              }
            }
            ++sfull;
            if (!(ok = __all_sync(0xffffffffu, ok))) break;   // the leader's warp leaves together
          }
          if (!ok) break;
        }
        if (!ok) break;
      }
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(acc_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      // dV first, released as soon as it is in registers and stored, then
      // dK (scaled by the softmax scale: dK = scale dS^T Q)
#pragma unroll
      for (int acc = 0; acc < 2; ++acc) {
        const uint32_t tcol = tmem + lane_off + (acc ? T_DK : T_DV);
        __nv_bfloat16* orow = acc ? dk_row : dv_row;
        const float mul = acc ? scale : 1.0f;
#pragma unroll
        for (int c = 0; c < (acc ? HD : HV) / 32; c += 2) {
          uint32_t v[2][32];
          ptx::tmem_ld32(tcol + c * 32, v[0]);
          ptx::tmem_ld32(tcol + c * 32 + 32, v[1]);
          ptx::tmem_ld_wait(v[0]);
          ptx::tmem_ld_wait(v[1]);
          if (key_ok) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                uint4 a;
                a.x = ptx::pack_bf16(__uint_as_float(v[h][8 * e + 0]) * mul, __uint_as_float(v[h][8 * e + 1]) * mul);
                a.y = ptx::pack_bf16(__uint_as_float(v[h][8 * e + 2]) * mul, __uint_as_float(v[h][8 * e + 3]) * mul);
                a.z = ptx::pack_bf16(__uint_as_float(v[h][8 * e + 4]) * mul, __uint_as_float(v[h][8 * e + 5]) * mul);
                a.w = ptx::pack_bf16(__uint_as_float(v[h][8 * e + 6]) * mul, __uint_as_float(v[h][8 * e + 7]) * mul);
                reinterpret_cast<uint4*>(orow + (c + h) * 32)[e] = a;
              }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(acc ? dk_free : dv_free);
      }
      ++u_it;
    }
    // every reduce issued by this CTA has landed before it exits
    if (ATOMIC_DQ && leader) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- deterministic dQ

// Every tile the dQ kernel reads passes through one FIFO ring of equal slots
// in the order it is consumed: per unit its Q, dO and O tiles, then K_0, V_0,
// K_1, V_1, ... of its key tiles. The row threads move Q and dO from their
// slots into tensor memory (and use dO and O for D = rowsum(dO o O)), after
// which the slots go back to the ring; Q and dO then serve from tensor memory
// as the A operands of S = Q K^T and dP = dO V^T. Each of the three products
// per key tile therefore reads only its B operand (a K or V tile) from shared
// memory: 96 KB of operand reads per key tile at d = dv = 128 instead of 160,
// and the slots Q and dO would occupy all unit long stream K and V instead.
template <int HD, int HV>
struct CfgQ {
  static constexpr int KB = HD / 64;          // 64-column boxes per Q / K row
  static constexpr int KBV = HV / 64;         // ... per V / dO / O row
  static constexpr int TILE = BT * HD * 2;    // one 128-row Q or K tile
  static constexpr int TILE_V = BT * HV * 2;  // one 128-row V, dO or O tile
  static constexpr int SLOT = TILE > TILE_V ? TILE : TILE_V;
  static constexpr int DPART_BYTES = 2 * 2 * BT * 4;   // [unit parity][row group][128] fp32 partial D
  static constexpr int NSLOT_FIT = (227 * 1024 - DPART_BYTES - 256) / SLOT;
  static constexpr int NSLOT = NSLOT_FIT < 16 ? NSLOT_FIT : 16;   // 7 at d = dv = 128
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_DPART = OFF_RING + NSLOT * SLOT;
  static constexpr int OFF_BAR = OFF_DPART + DPART_BYTES;
  // full[NSLOT], empty[NSLOT], qd_ready, s_full, s_free, dp_full, ds_full, dq_full, drain, dpart_full,
  // unit queue full[4], empty[4]
  static constexpr int NBAR = 2 * NSLOT + 8 + 2 * UnitQueue::N;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM address, abort word, unit queue slots
  static constexpr int SMEM = OFF_MISC + 16 + 4 * UnitQueue::N;
  static constexpr int UQ_READERS = 1 + 256;   // the MMA warp (once) and every row thread
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16(BT, BT, false, false);    // S, dP (A in TMEM)
  static constexpr uint32_t IDESC_DQ = ptx::idesc_bf16(BT, HD, false, true);    // dQ (A in TMEM, K MN-major)
  // TMEM columns: Q and dO as packed bf16 (two elements per column), the S
  // and dP tiles (fp32; dS is packed over the first half of each group's dP
  // columns), the dQ accumulator
  static constexpr uint32_t T_Q = 0, T_DO = 64, T_S = 128, T_DP = 256, T_DQ = 384;
  static_assert(HD / 2 <= 64 && HV / 2 <= 64 && T_DQ + HD <= 512, "TMEM columns");
};
constexpr int DQ_THREADS = 320;

// One persistent CTA per SM; a unit is one 128-row query tile of one head.
// Per unit the row threads stage Q and dO into TMEM and form the tile's D =
// rowsum(dO o O) and -LSE * log2(e), which they use and store for the dK/dV
// kernel that runs after this one. Then, for each key tile (fixed ascending
// order): S = Q K^T and dP = dO V^T (both in TMEM), dS = P o (dP - D) written
// bf16 over dP, and dQ += dS K accumulates in TMEM. Per key tile j the MMA
// warp issues S_{j+1}, dQ_j, dP_{j+1}: the next scores are computed while the
// row threads turn dP_j into dS_j, and dP_{j+1} overwrites the dP tile only
// after dQ_j has read dS_j (MMAs of one thread run in issue order).
// Warps: 0 producer, 1 MMA, 2-5 and 6-9 two row groups; group g works on key
// columns [64g, 64g + 64) of every query row (one thread per row each), packs
// its dS at columns [64g, 64g + 32) of the dP tile, and stages columns
// [g d/2, (g + 1) d/2) of Q (and of dO) into TMEM.
// SPLIT: key ranges per unit, fp32 partial dQ (see Params).
template <int HD, int HV, bool SPLIT>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ CUtensorMap tmO, const Params P) {
  using C = CfgQ<HD, HV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  uint8_t* ring = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;                   // [NSLOT]
  uint64_t* empty = full + C::NSLOT;       // [NSLOT]
  uint64_t* qd_ready = empty + C::NSLOT;   // the row threads staged a unit's Q and dO (and read its O)
  uint64_t* s_full = qd_ready + 1;
  uint64_t* s_free = qd_ready + 2;
  uint64_t* dp_full = qd_ready + 3;
  uint64_t* ds_full = qd_ready + 4;
  uint64_t* dq_full = qd_ready + 5;
  uint64_t* drain = qd_ready + 6;
  uint64_t* dpart_full = qd_ready + 7;     // both row groups have written a unit's partial D
  float* dpart = reinterpret_cast<float*>(smem + C::OFF_DPART);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  const UnitQueue uq{reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16), qd_ready + 8,
                     qd_ready + 8 + UnitQueue::N};
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(full + s, 1);
      ptx::mbar_init(empty + s, 1);
    }
    for (int s = 0; s < UnitQueue::N; ++s) {
      ptx::mbar_init(uq.full + s, 1);
      ptx::mbar_init(uq.empty + s, C::UQ_READERS);
    }
    ptx::mbar_init(qd_ready, 256);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_free, 256);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(ds_full, 256);
    ptx::mbar_init(dq_full, 1);
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(dpart_full, 256);
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
  const int Tq = P.p.Tq, Tk = P.p.Tk;
  // the launch's units: (query tile, key split) blocks of every head, handed
  // out at run time in head groups, the longest (causal: last) blocks first
  const int nb = P.n_q_tiles * P.dq_splits, nh = P.p.B * P.p.H, total = nb * nh;
  const int cta = blockIdx.x, grid = gridDim.x;
  auto decode = [&](int x, int* bh, int* blk) { grouped_unit(x, nb, nh, P.group, P.p.causal != 0, bh, blk); };
  // Ring item i (counted across units) sits in slot i % NSLOT. A unit whose
  // first item is i0 has Q at i0, dO at i0 + 1, O at i0 + 2, and K_j, V_j of
  // its j-th key tile at i0 + 3 + 2j and i0 + 4 + 2j.
  auto slot = [](uint32_t i) { return static_cast<int>(i % C::NSLOT); };
  auto par = [](uint32_t i) { return (i / C::NSLOT) & 1u; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::WaitCtx w{abort_flag, P.status, 5u};
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
    ptx::tma_prefetch_desc(&tmdO);
    ptx::tma_prefetch_desc(&tmO);
    uint32_t item = 0, pu = 0;
    int bh = 0, blk = 0;
    auto load = [&](const CUtensorMap* map, int boxes, uint32_t bytes, int row) {
      const int s = slot(item);
      if (!ptx::mbar_wait(empty + s, par(item) ^ 1u, w)) return false;
      ptx::mbar_arrive_expect_tx(full + s, bytes);
      for (int b = 0; b < boxes; ++b) ptx::tma_load_3d(ring + s * C::SLOT + b * BOX_BYTES, map, full + s, b * 64, row, bh);
      ++item;
      return true;
    };
    // take the next unit and publish it; the next one is published before
    // this one's tiles are loaded, so that the row threads can stage it
    // while they finish this one
    int x = next_unit_index(P, pu, cta, grid, total);
    bool ok = !P.dynamic || uq_push(uq, pu, x, w);
    ++pu;
    while (ok && x < total) {
      const int xn = next_unit_index(P, pu, cta, grid, total);
      if (P.dynamic && !(ok = uq_push(uq, pu, xn, w))) break;
      ++pu;
      decode(x, &bh, &blk);
      x = xn;
      int qt, sp_, j0, nk;
      if (!dq_unit<SPLIT>(P, blk, &qt, &sp_, &j0, &nk)) continue;
      ok = load(&tmQ, C::KB, C::TILE, qt * BT) && load(&tmdO, C::KBV, C::TILE_V, qt * BT) &&
           load(&tmO, C::KBV, C::TILE_V, qt * BT);
      for (int j = 0; ok && j < nk; ++j)
        ok = load(&tmK, C::KB, C::TILE, (j0 + j) * BT) && load(&tmV, C::KBV, C::TILE_V, (j0 + j) * BT);
    }
    if (!ok) {
      // Let the copies already in flight land before the CTA exits: each of
      // the last NSLOT items issued is the latest load of its slot.
      for (uint32_t n = (item > static_cast<uint32_t>(C::NSLOT) ? item - C::NSLOT : 0u); n < item; ++n)
        ptx::mbar_wait_drain(full + slot(n), par(n));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp follows the schedule and waits; the elected lane (lane 0)
    // issues the MMAs and commits (see the dK/dV kernel).
    ptx::WaitCtx w{abort_flag, P.status, 6u};
    const uint32_t aR = ptx::smem_u32(ring);
    auto kmaj = [](uint32_t base, int kk) {
      return ptx::sdesc_advance(ptx::sdesc_sw128(base, 16, 1024), (kk >> 2) * BOX_BYTES + (kk & 3) * 32);
    };
    auto mnmaj = [](uint32_t base, int kk) {
      return ptx::sdesc_advance(ptx::sdesc_sw128(base, BOX_BYTES, 1024), kk * 2048);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    auto mma_s = [&](uint32_t ik) {   // S = Q K^T: Q from TMEM (8 columns per 16 of d), K tile of item ik
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        ptx::mma_ts(tmem + C::T_S, tmem + C::T_Q + 8 * kk, kmaj(aR + slot(ik) * C::SLOT, kk), C::IDESC_S, kk > 0);
      ptx::mma_commit(s_full);
    };
    auto mma_dp = [&](uint32_t iv) {   // dP = dO V^T: dO from TMEM, V tile of item iv (read by nothing later)
#pragma unroll
      for (int kk = 0; kk < HV / 16; ++kk)
        ptx::mma_ts(tmem + C::T_DP, tmem + C::T_DO + 8 * kk, kmaj(aR + slot(iv) * C::SLOT, kk), C::IDESC_S,
                    kk > 0);
      ptx::mma_commit(dp_full);
      ptx::mma_commit(empty + slot(iv));
    };
    uint32_t item = 0, u_it = 0, sp = 0, ru = 0;
    bool ok = true, moved = false;
    int bh, blk;
    while (ok) {
      int x;
      if (P.dynamic) {
        if (!(ok = uq_read(uq, ru, &x, w))) break;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(uq.empty + ru % UnitQueue::N);
      } else {
        x = next_unit_index(P, ru, cta, grid, total);
      }
      ++ru;
      if (x >= total) break;
      decode(x, &bh, &blk);
      int qt, sp_, j0, nk;
      if (!dq_unit<SPLIT>(P, blk, &qt, &sp_, &j0, &nk)) continue;
      const uint32_t i0 = item;
      // Q and dO are in TMEM and the row threads are done with the three
      // staging slots, which go back to the ring
      if (!(ok = wait(qd_ready, u_it & 1u))) break;
      if (lane == 0)
        for (int k = 0; k < 3; ++k) ptx::mbar_arrive(empty + slot(i0 + k));
      __syncwarp();
      // S and dP of the first key tile
      if (!(ok = wait(full + slot(i0 + 3), par(i0 + 3)))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        mma_s(i0 + 3);
      }
      __syncwarp();
      if (!(ok = wait(full + slot(i0 + 4), par(i0 + 4)))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        mma_dp(i0 + 4);
      }
      __syncwarp();
      // K of the next key tile: each step waits for the tiles of the step
      // after it while its own MMAs run
      if (nk > 1 && !(ok = wait(full + slot(i0 + 5), par(i0 + 5)))) break;
      for (int j = 0; j < nk; ++j, ++sp) {
        const uint32_t ik = i0 + 3 + 2 * j;   // K_j; V_{j+1} = ik + 3, K_{j+1} = ik + 2, K_{j+2} = ik + 4
        if (j + 1 < nk) {
          // S of the next key tile once the row threads hold this one in registers
          if (!(ok = wait(s_free, sp & 1u))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_s(ik + 2);
          }
          __syncwarp();
        }
        // dQ += dS K
        if (!(ok = wait(ds_full, sp & 1u))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)
            ptx::mma_ts(tmem + C::T_DQ, tmem + C::T_DP + packed_col(kk), mnmaj(aR + slot(ik) * C::SLOT, kk),
                        C::IDESC_DQ, (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(empty + slot(ik));
        }
        __syncwarp();
        if (j + 1 < nk) {
          // dP of the next key tile, into the tile dQ_j has just been given
          if (!(ok = wait(full + slot(ik + 3), par(ik + 3)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_dp(ik + 3);
          }
          __syncwarp();
        }
        if (j + 2 < nk && !(ok = wait(full + slot(ik + 4), par(ik + 4)))) break;
      }
      if (!ok) break;
      if (ptx::elect_one()) {
        moved |= lane != 0;
        ptx::mma_commit(dq_full);
      }
      __syncwarp();
      item = i0 + 3 + 2 * nk;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ row groups
    const int g = (warp - 2) >> 2;          // row group: key columns [64g, 64g + 64)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S + 64 * g, tDP = tmem + lane_off + C::T_DP + 64 * g;
    const uint32_t tDQ = tmem + lane_off + C::T_DQ + (HD / 2) * g;
    const uint32_t tQ = tmem + lane_off + C::T_Q + (HD / 4) * g, tDO = tmem + lane_off + C::T_DO + (HV / 4) * g;
    ptx::WaitCtx w{abort_flag, P.status, 7u + g};
    const float sc2 = P.sc2, scale = P.p.scale;
    // Stage the unit whose first ring item is i0 (the u-th unit of this CTA):
    // this group's half of row r of Q and of dO into TMEM, and its half of
    // D_r = sum_c dO_rc O_rc ("attention_backprop", section "Gradient of S":
    // ROW_SUM(dL/dO o O)) into dpart. Rows past Tq load as zeros.
    auto stage = [&](uint32_t i0, uint32_t u) {
      for (int k = 0; k < 3; ++k)
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(full + slot(i0 + k), par(i0 + k), w))) return false;
      const uint8_t* sq = ring + slot(i0) * C::SLOT;
      const uint8_t* sdo = ring + slot(i0 + 1) * C::SLOT;
      const uint8_t* so = ring + slot(i0 + 2) * C::SLOT;
      {
        uint32_t v[HD / 4];
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint4 x = *reinterpret_cast<const uint4*>(sq + sw128_offset(r, (HD / 2) * g + 8 * k));
          v[4 * k] = x.x;
          v[4 * k + 1] = x.y;
          v[4 * k + 2] = x.z;
          v[4 * k + 3] = x.w;
        }
        if constexpr (HD == 128) ptx::tmem_st32(tQ, v); else ptx::tmem_st16(tQ, v);
      }
      float part = 0.f;
      {
        uint32_t v[HV / 4];
#pragma unroll
        for (int k = 0; k < HV / 16; ++k) {
          const uint32_t off = sw128_offset(r, (HV / 2) * g + 8 * k);
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
      ptx::mbar_arrive(qd_ready);
      return true;
    };
    // the CTA's next unit with at least one key tile: 1, or 0 at the end of
    // the launch's units, -1 on a timeout
    uint32_t ru = 0;
    auto next_unit = [&](int* bh, int* qt, int* split, int* j0, int* nk) {
      for (;;) {
        int x, bl;
        if (P.dynamic) {
          if (!uq_read(uq, ru, &x, w)) return -1;
          ptx::mbar_arrive(uq.empty + ru % UnitQueue::N);
        } else {
          x = next_unit_index(P, ru, cta, grid, total);
        }
        ++ru;
        if (x >= total) return 0;
        decode(x, bh, &bl);
        if (dq_unit<SPLIT>(P, bl, qt, split, j0, nk)) return 1;
      }
    };
    uint32_t item = 0, u_it = 0, sp = 0;
    int bh, qt, split, j0, nk;
    const int first = next_unit(&bh, &qt, &split, &j0, &nk);
    bool have = first == 1;
    bool ok = first >= 0 && (!have || stage(0u, 0u));
    while (ok && have) {
      const int q = qt * BT + r;
      const bool q_ok = q < Tq;
      const float lse = q_ok ? P.LSE[static_cast<size_t>(bh) * Tq + q] : -CUDART_INF_F;
      const float nlse2 = (lse == -CUDART_INF_F) ? -CUDART_INF_F : -lse * LOG2E;
      // D of this unit: the two groups' halves (padding rows get D = 0 and
      // -LSE * log2(e) = -inf, so their P and dS are 0)
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dpart_full, u_it & 1u, w)))) break;
      const float* dpu = dpart + (u_it & 1u) * 2 * BT;
      const float dd = dpu[r] + dpu[BT + r];
      // stored for every row of the padded tile: the dK/dV kernel reads whole
      // 128-row slices, and its padding rows must hold D = 0, -inf
      if (g == 0 && split == 0) {   // (every split forms the same D)
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
          for (int c = 0; c < 2; ++c) ptx::tmem_ld32(tS + c * 32, v[c]);   // both in flight
#pragma unroll
          for (int c = 0; c < 2; ++c) ptx::tmem_ld_wait(v[c]);
          // S is in registers: the next S product may overwrite it while the
          // exponentials below run
          ptx::tc_fence_before();
          ptx::mbar_arrive(s_free);
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
        for (int c = 0; c < 2; ++c) ptx::tmem_ld32(tDP + c * 32, v[c]);   // both in flight
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
          // packed over this group's own first 32 columns (already read)
          ptx::tmem_st16(tDP + c * 16, pk);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ds_full);
      }
      if (!ok) break;
      // The next unit's Q and dO go into TMEM now: the S and dP products that
      // read this unit's have completed (their results were consumed above),
      // so the next unit's first S can start while this unit's epilogue runs.
      const uint32_t i_next = item + 3 + 2 * nk;
      int nbh = 0, nqt = 0, nsplit = 0, nj0 = 0, nnk = 0;
      const int nx = next_unit(&nbh, &nqt, &nsplit, &nj0, &nnk);
      ok = nx >= 0;
      if (!ok) break;
      const bool have_next = nx == 1;
      if (have_next && !(ok = stage(i_next, u_it + 1))) break;
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dq_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      // this group writes dQ columns [g HD / 2, (g + 1) HD / 2) of its row
      if (SPLIT) {
        const size_t rows = static_cast<size_t>(P.p.B) * P.p.H * Tq;
        float* prow = P.dQpart + (static_cast<size_t>(split) * rows + static_cast<size_t>(bh) * Tq + (q_ok ? q : 0)) *
                                     HD + (HD / 2) * g;
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
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
        __nv_bfloat16* row = P.dQ + (static_cast<size_t>(bh) * Tq + (q_ok ? q : 0)) * HD + (HD / 2) * g;
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
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
      // waits for this group's first dS of that unit, issued after this)
      ptx::tc_fence_before();
      item = i_next;
      ++u_it;
      have = have_next;
      bh = nbh;
      qt = nqt;
      split = nsplit;
      j0 = nj0;
      nk = nnk;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// dQ (bf16) = the sum of the split dQ kernel's partials (fp32, already
// scaled) in split order, over the splits that hold key tiles of the row's
// query tile; one thread per 4 columns of a row.
__global__ void reduce_dq_kernel(const float* __restrict__ part, uint2* __restrict__ out, long long rows, int Tq,
                                 int d, int n_splits, int split_tiles, int n_k_tiles, int causal) {
  const long long n4 = rows * (d / 4);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const long long r = i / (d / 4);
    const int qt = static_cast<int>(r % Tq) / BT;
    const int nt = causal ? min(qt + 1, n_k_tiles) : n_k_tiles;
    const int ns = min(n_splits, (nt + split_tiles - 1) / split_tiles);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
      const float4 v = reinterpret_cast<const float4*>(part)[static_cast<long long>(s) * n4 + i];
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    out[i] = make_uint2(ptx::pack_bf16(a.x, a.y), ptx::pack_bf16(a.z, a.w));
  }
}

// dQ (bf16) = dQ accumulator (fp32, already scaled)
__global__ void convert_dq_kernel(const float4* __restrict__ acc, uint2* __restrict__ out, size_t n4) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = acc[i];
    out[i] = make_uint2(ptx::pack_bf16(v.x, v.y), ptx::pack_bf16(v.z, v.w));
  }
}

template <int HD, int HV>
cudaError_t launch(const LaunchBwd& a) {
  const Problem& p = a.p;
  const bool atomic = !a.deterministic;
  // Deterministic: the dQ kernel forms D and -LSE * log2(e) itself and runs
  // before the dK/dV kernel, which reads them; there is no preprocess.
  const bool pre = atomic && (a.phase == 0 || a.phase == 1), conv = a.phase == 0 || a.phase == 3;
  const bool main_kv = a.phase == 0 || a.phase == 2 || a.phase == 4;
  const bool main_q = a.phase == 0 || a.phase == 2 || a.phase == 5;
  // Phase 6: the dQ pass on CTA pairs (dq_pair.cu, d = 128), in place of
  // phase 5. It halves each SM's K and V operand traffic but adds a cross-SM
  // handshake to every key step; at B=2 H=16 T=8192 d=128 causal it measured
  // 0.539 ms against 0.500 ms for the one-CTA kernel, which attn_bwd runs.
  const bool pairs_q = a.phase == 6;
  cudaError_t e = cudaSuccess;
  if (pre) {
    e = launch_bwd_preprocess(p, a.O, a.dO, a.LSE, 2, a.D, a.NLSE2, atomic ? a.dQacc : nullptr, p.d, a.num_sms,
                              a.stream);
    if (e != cudaSuccess) return e;
  }
  Params P{};
  P.p = p;
  P.NLSE2 = a.NLSE2;
  P.D = a.D;
  P.LSE = a.LSE;
  P.Tq_pad = padded_rows(p.Tq);
  P.dQacc = a.dQacc;
  P.dQ = static_cast<__nv_bfloat16*>(a.dQ);
  P.dK = static_cast<__nv_bfloat16*>(a.dK);
  P.dV = static_cast<__nv_bfloat16*>(a.dV);
  P.status = a.status;
  P.n_q_tiles = (p.Tq + BT - 1) / BT;
  P.n_k_tiles = (p.Tk + BT - 1) / BT;
  P.sc2 = p.scale * LOG2E;
  const int heads = p.B * p.H;
  const bool split_dq = !atomic && a.dq_splits > 1;
  // Unit order of the dQ and dK/dV kernels. When the tiles a kernel streams
  // (K and V of every head for the dQ kernel, Q, dO and the LSE / D slices
  // for the dK/dV kernel) exceed L2 twice over, the units are claimed at run
  // time from a counter (zeroed before the launch) in head groups whose tiles
  // fill about half of L2, so that each group's tiles are read from DRAM
  // about once; otherwise each CTA takes its static share of all heads,
  // heaviest first (measured on GB300, fwd+bwd: B=1 H=32 T=32768 d=128
  // 1164-1218 -> 1280-1297 TFLOP/s with the groups, DRAM reads per launch of
  // the dQ kernel 38.7 -> 2.0 GB and of the dK/dV kernel 24.2 -> 1.1 GB;
  // B=2 H=16 T=8192 needs no groups and is unchanged; B=4 H=16 T=2048 was
  // slower with run-time claiming, 547 -> 526).
  P.sched = a.sched;
  auto heads_per_group = [&](size_t per_head) {
    if (per_head * heads <= 2 * a.l2_bytes) return heads;
    const size_t budget = a.l2_bytes / 2;
    size_t g = per_head ? budget / per_head : heads;
    if (g < 1) g = 1;
    if (g > static_cast<size_t>(heads)) g = heads;
    return static_cast<int>(g);
  };
  const int group_q = heads_per_group(static_cast<size_t>(p.Tk) * (p.d + p.dv) * 2);
  const int group_kv = heads_per_group(static_cast<size_t>(p.Tq) * (p.d + p.dv) * 2 + P.Tq_pad * 8ull);
  P.dq_splits = split_dq ? a.dq_splits : 1;
  P.dq_split_tiles = split_dq ? a.dq_split_tiles : P.n_k_tiles;
  P.dQpart = a.dQpart;
  if (pairs_q) {
    if (atomic || HD != 128) return cudaErrorInvalidValue;   // (the host checks this first)
    if ((e = launch_dq_pair(a, P)) != cudaSuccess) return e;
  } else if (!atomic && main_q) {
    if (static_cast<long long>(P.n_q_tiles) * P.dq_splits * heads > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int units = P.n_q_tiles * P.dq_splits * heads;
    P.dynamic = group_q < heads;
    // the static order: heaviest first over all heads (causal), head by head (no mask)
    P.group = P.dynamic ? group_q : (p.causal ? heads : 1);
    if (P.dynamic && (e = cudaMemsetAsync(a.sched, 0, sizeof(uint32_t), a.stream)) != cudaSuccess) return e;
    const int grid = units < a.num_sms ? units : a.num_sms;
    using CQ = CfgQ<HD, HV>;
    static_assert(CQ::SMEM <= 227 * 1024, "shared memory");
    auto kern = split_dq ? dq_kernel<HD, HV, true> : dq_kernel<HD, HV, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CQ::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, DQ_THREADS, CQ::SMEM, a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, *a.tmdO, *a.tmO, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (main_kv) {
    P.order = Order{P.n_k_tiles, heads, p.causal ? 2 : 0};   // the static order
    const int units = P.n_k_tiles * heads;
    P.sched = a.sched + 1;
    P.dynamic = group_kv < heads;
    P.group = P.dynamic ? group_kv : (p.causal ? heads : 1);
    if (P.dynamic && (e = cudaMemsetAsync(P.sched, 0, sizeof(uint32_t), a.stream)) != cudaSuccess) return e;
    const int grid = units < a.num_sms ? units : a.num_sms;
    static_assert(CfgKV<HD, HV, true>::SMEM <= 227 * 1024 && CfgKV<HD, HV, false>::SMEM <= 227 * 1024,
                  "shared memory");
    auto kern = atomic ? (P.dynamic ? dkdv_kernel<HD, HV, true, true> : dkdv_kernel<HD, HV, true, false>)
                       : (P.dynamic ? dkdv_kernel<HD, HV, false, true> : dkdv_kernel<HD, HV, false, false>);
    const int smem = atomic ? CfgKV<HD, HV, true>::SMEM : CfgKV<HD, HV, false>::SMEM;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // The register split must fit the launch allocation (see reg_acquire).
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    const int split = atomic ? KvRegs<true>::CTRL + 2 * KvRegs<true>::PDS + KvRegs<true>::DQ
                             : KvRegs<false>::CTRL + 2 * KvRegs<false>::PDS + KvRegs<false>::DQ;
    if (fa.numRegs != KV_REG_LAUNCH || split > 4 * KV_REG_LAUNCH)
      return cudaErrorInvalidConfiguration;
    kern<<<grid, KV_THREADS, smem, a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, *a.tmdO,
                                                           atomic ? *a.tmdQacc : *a.tmQ, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (split_dq && conv) {
    const long long rows = static_cast<long long>(heads) * p.Tq;
    reduce_dq_kernel<<<a.num_sms * 8, 256, 0, a.stream>>>(a.dQpart, static_cast<uint2*>(a.dQ), rows, p.Tq, p.d,
                                                          P.dq_splits, P.dq_split_tiles, P.n_k_tiles, p.causal);
    return cudaGetLastError();
  }
  if (atomic) {
    if (!conv) return cudaSuccess;
    const size_t n4 = static_cast<size_t>(heads) * p.Tq * p.d / 4;
    convert_dq_kernel<<<a.num_sms * 4, 256, 0, a.stream>>>(reinterpret_cast<const float4*>(a.dQacc),
                                                            static_cast<uint2*>(a.dQ), n4);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace bwd

cudaError_t launch_bwd_bf16(const LaunchBwd& a) {
  if (a.p.d == 128) return a.p.dv == 128 ? bwd::launch<128, 128>(a) : bwd::launch<128, 64>(a);
  return a.p.dv == 128 ? bwd::launch<64, 128>(a) : bwd::launch<64, 64>(a);
}

}  // namespace attn
