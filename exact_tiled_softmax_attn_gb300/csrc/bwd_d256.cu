// bf16 attention backward for d = 256 on tcgen05 tensor cores (sm_103a).
//
// The gradients of "attention_backprop" (sections "Gradient of V and P",
// "Gradient of S", "Gradient of Q and K"), P recomputed tile by tile from the
// stored log-sum-exp ("The Hidden Recurrence in Softmax Attention", section
// "Flash Attention Backward Pass"):
//   P = exp(scale Q K^T - LSE), dV = P^T dO, dP = dO V^T, dS = P o (dP - D),
//   dK = scale dS^T Q, dQ = scale dS K,  D = rowsum(dO o O) (formed by the dQ kernel).
// With rows of 256 columns the dK and dV accumulators of one 128-key tile
// fill tensor memory's 512 columns on their own, so the work is split into
// three kernels, each of which holds one accumulator next to its score tiles:
//   kv256_kernel<DV, 0>  per 128-key tile: S^T = K Q^T, P^T, dV += P^T dO
//   kv256_kernel<DV, 1>  per 128-key tile: S^T, dP^T = V dO^T, dS^T, dK += dS^T Q
//   q256_kernel<DV>      per 128-row query tile: D, then S = Q K^T, dP = dO V^T, dS, dQ += dS K
// The dQ kernel runs first and stores D and -LSE log2(e) for the other two.
// The key-tile kernels walk the query rows in steps of 64 and the query-tile
// kernel the keys in steps of 64, so that the 256-column accumulator, the
// 128 columns of the resident operand (K or Q as packed bf16, the A operand
// of the score product) and the step's 64-column score tiles fit together.
// Every accumulation runs in a fixed order: the results are bitwise
// reproducible.
//
// Warps (320 threads): 0 producer (lane 0: TMA and bulk copies), 1 MMA issuer
// (elected lane; allocates and frees TMEM), 2-5 and 6-9 two row groups: one
// thread per row of the 128-row tile, group g on columns [32g, 32g + 32) of
// each 64-wide step. Streamed tiles pass through one FIFO ring of 32 KB slots
// as 64-row TMA boxes (64 x 64 bf16 each, 128-byte swizzle).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "bwd_common.cuh"
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace bwd256 {

using bwd::BT;
using bwd::LOG2E;
using bwd::Order;
using bwd::Params;

constexpr int HD = 256;                   // d
constexpr int NS = 64;                    // rows (queries or keys) per step
constexpr int BOX64 = 64 * 64 * 2;        // one TMA box: 64 rows x 64 bf16
constexpr int BOX128 = 128 * 64 * 2;      // one TMA box: 128 rows x 64 bf16
constexpr int SLOT = 64 * HD * 2;         // 32 KB: 64 rows of Q or K (or of dO / V, dv <= 256)
constexpr int THREADS = 320;

// K-major operand of 64 (or 128) rows stored as 64-column boxes `box` bytes
// apart, k-step kk of 16 elements.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int box, int kk) {
  return ptx::sdesc_advance(ptx::sdesc_sw128(base, 16, 1024), (kk >> 2) * box + (kk & 3) * 32);
}
// MN-major operand of 64 rows (the K dimension) whose N columns are 64-column
// boxes of BOX64 bytes, k-step kk of 16 rows.
__device__ __forceinline__ uint64_t mnmaj64(uint32_t base, int kk) {
  return ptx::sdesc_advance(ptx::sdesc_sw128(base, BOX64, 1024), kk * 2048);
}

// --------------------------------------------------------------------------
// Key-tile kernels. MODE 0: dV; MODE 1: dK.

template <int DV, int MODE>
struct CfgKV {
  static constexpr int VRES = MODE == 1 ? BT * DV * 2 : 0;   // V of the unit (A operand of dP^T), 128-row boxes
  static constexpr int NL = 4;                               // slots of -LSE*log2(e) / D slices
  static constexpr int LBYTES = 2 * NS * 4;                  // one slice slot: 64 + 64 fp32
  static constexpr int NSLOT_FIT = (227 * 1024 - VRES - NL * LBYTES - 512) / SLOT;
  static constexpr int NSLOT = NSLOT_FIT < 16 ? NSLOT_FIT : 16;
  static constexpr int OFF_V = 0;
  static constexpr int OFF_RING = OFF_V + VRES;
  static constexpr int OFF_L = OFF_RING + NSLOT * SLOT;
  static constexpr int OFF_BAR = OFF_L + NL * LBYTES;
  // full[NSLOT], empty[NSLOT], l_full[NL], l_empty[NL], k_ready, v_full, v_empty, s_full[2], s_free,
  // p_full[2], dp_full, ds_full, acc_full, acc_free, drain
  static constexpr int NBAR = 2 * NSLOT + 2 * NL + 14;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t IDESC_ST = ptx::idesc_bf16(BT, NS, false, false);   // S^T, dP^T: N = 64 queries
  static constexpr uint32_t IDESC_ACC = ptx::idesc_bf16(BT, MODE == 0 ? DV : HD, false, true);   // dV or dK
  // TMEM columns: K (packed bf16, 128), score tiles, accumulator at 256
  static constexpr uint32_t T_K = 0, T_S = 128, T_DP = 192, T_ACC = 256;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NSLOT >= 4, "ring");
};

// Query steps of key tile kb: from the first 64-row step that can see it
// (causal) to the last step holding rows below Tq.
__device__ __forceinline__ void kv_steps(const Params& P, int kb, int* t0, int* nt) {
  const int last = (P.p.Tq + NS - 1) / NS;
  *t0 = P.p.causal ? 2 * kb : 0;
  *nt = last > *t0 ? last - *t0 : 0;
}

template <int DV, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    kv256_kernel(const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ CUtensorMap tmK64,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO64,
                 const Params P) {
  using C = CfgKV<DV, MODE>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* ring = smem + C::OFF_RING;
  float* sL = reinterpret_cast<float*>(smem + C::OFF_L);   // [NL][2][64]: -LSE*log2(e), D
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;                      // [NSLOT]
  uint64_t* empty = full + C::NSLOT;          // [NSLOT]
  uint64_t* l_full = empty + C::NSLOT;        // [NL]
  uint64_t* l_empty = l_full + C::NL;         // [NL]
  uint64_t* k_ready = l_empty + C::NL;        // the row threads staged the unit's K into TMEM
  uint64_t* v_full = k_ready + 1;
  uint64_t* v_empty = k_ready + 2;
  uint64_t* s_full = k_ready + 3;             // [2] by step parity (MODE 0); [0] only (MODE 1)
  uint64_t* s_free = k_ready + 5;             // MODE 1: the row threads hold S^T in registers
  uint64_t* p_full = k_ready + 6;             // [2] MODE 0: P^T written over the step's S^T tile
  uint64_t* dp_full = k_ready + 8;
  uint64_t* ds_full = k_ready + 9;            // MODE 1: dS^T written over dP^T
  uint64_t* acc_full = k_ready + 10;
  uint64_t* acc_free = k_ready + 11;          // the epilogue has read the accumulator
  uint64_t* drain = k_ready + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(full + s, 1);
      ptx::mbar_init(empty + s, 1);
    }
    for (int s = 0; s < C::NL; ++s) {
      ptx::mbar_init(l_full + s, 1);
      ptx::mbar_init(l_empty + s, 256);
    }
    ptx::mbar_init(k_ready, 256);
    ptx::mbar_init(v_full, 1);
    ptx::mbar_init(v_empty, 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(s_full + b, 1);
      ptx::mbar_init(p_full + b, 256);
    }
    ptx::mbar_init(s_free, 256);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(ds_full, 256);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_free, 256);
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
  const int Tk = P.p.Tk;
  // Ring item i (counted across units) sits in slot i % NSLOT. A unit whose
  // first item is i0 has its K tile's halves at i0, i0 + 1, then per query
  // step t the 64 rows of Q at i0 + 2 + 2t and of dO at i0 + 3 + 2t. Query
  // step number n (counted across units) uses slice slot n % NL.
  auto slot = [](uint32_t i) { return static_cast<int>(i % C::NSLOT); };
  auto par = [](uint32_t i) { return (i / C::NSLOT) & 1u; };
  auto lslot = [](uint32_t n) { return static_cast<int>(n % C::NL); };
  auto lpar = [](uint32_t n) { return (n / C::NL) & 1u; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::WaitCtx w{abort_flag, P.status, 21u};
    ptx::tma_prefetch_desc(&tmQ64);
    ptx::tma_prefetch_desc(&tmK64);
    ptx::tma_prefetch_desc(&tmdO64);
    if (MODE == 1) ptx::tma_prefetch_desc(&tmV);
    uint32_t item = 0, n = 0, u_it = 0, l_issued = 0, v_issued = 0;
    bool ok = true;
    int bh, kb;
    auto load = [&](const CUtensorMap* map, int boxes, uint32_t bytes, int row) {
      const int s = slot(item);
      if (!ptx::mbar_wait(empty + s, par(item) ^ 1u, w)) return false;
      ptx::mbar_arrive_expect_tx(full + s, bytes);
      for (int b = 0; b < boxes; ++b) ptx::tma_load_3d(ring + s * SLOT + b * BOX64, map, full + s, b * 64, row, bh);
      ++item;
      return true;
    };
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &kb); ++round) {
      int t0, nt;
      kv_steps(P, kb, &t0, &nt);
      if (nt == 0) continue;
      ok = load(&tmK64, HD / 64, 64 * HD * 2, kb * BT) && load(&tmK64, HD / 64, 64 * HD * 2, kb * BT + 64);
      if (ok && MODE == 1) {
        // V of the unit, once the previous unit's last dP^T product has read it
        if (!(ok = ptx::mbar_wait(v_empty, (u_it & 1u) ^ 1u, w))) break;
        ptx::mbar_arrive_expect_tx(v_full, BT * DV * 2);
        for (int b = 0; b < DV / 64; ++b) ptx::tma_load_3d(sV + b * BOX128, &tmV, v_full, b * 64, kb * BT, bh);
        v_issued = u_it + 1;
      }
      for (int t = 0; ok && t < nt; ++t, ++n) {
        const int q0 = (t0 + t) * NS;
        const int ls = lslot(n);
        if (!(ok = ptx::mbar_wait(l_empty + ls, lpar(n) ^ 1u, w))) break;
        const size_t row0 = static_cast<size_t>(bh) * P.Tq_pad + q0;   // (q0 + 64 <= Tq_pad)
        ptx::mbar_arrive_expect_tx(l_full + ls, (MODE == 1 ? 2 : 1) * NS * 4);
        ptx::bulk_load(sL + ls * 2 * NS, P.NLSE2 + row0, NS * 4, l_full + ls);
        if (MODE == 1) ptx::bulk_load(sL + ls * 2 * NS + NS, P.D + row0, NS * 4, l_full + ls);
        l_issued = n + 1;
        ok = load(&tmQ64, HD / 64, 64 * HD * 2, q0) && load(&tmdO64, DV / 64, 64 * DV * 2, q0);
      }
      ++u_it;
    }
    if (!ok) {
      for (uint32_t m = (item > static_cast<uint32_t>(C::NSLOT) ? item - C::NSLOT : 0u); m < item; ++m)
        ptx::mbar_wait_drain(full + slot(m), par(m));
      for (uint32_t m = (l_issued > static_cast<uint32_t>(C::NL) ? l_issued - C::NL : 0u); m < l_issued; ++m)
        ptx::mbar_wait_drain(l_full + lslot(m), lpar(m));
      if (v_issued > 0) ptx::mbar_wait_drain(v_full, (v_issued - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    ptx::WaitCtx w{abort_flag, P.status, 22u};
    const uint32_t aR = ptx::smem_u32(ring), aV = ptx::smem_u32(sV);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    // S^T = K Q^T into score tile `col`: K from TMEM, the Q rows of item iq
    auto mma_st = [&](uint32_t iq, uint32_t col) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        ptx::mma_ts(tmem + col, tmem + C::T_K + 8 * kk, kmaj(aR + slot(iq) * SLOT, BOX64, kk), C::IDESC_ST, kk > 0);
    };
    uint32_t item = 0, u_it = 0, gs = 0;
    bool ok = true, moved = false;
    int bh, kb;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &kb); ++round) {
      int t0, nt;
      kv_steps(P, kb, &t0, &nt);
      if (nt == 0) continue;
      const uint32_t i0 = item;
      // K is in TMEM; its two staging slots go back to the ring
      if (!(ok = wait(k_ready, u_it & 1u))) break;
      if (lane == 0) {
        ptx::mbar_arrive(empty + slot(i0));
        ptx::mbar_arrive(empty + slot(i0 + 1));
      }
      __syncwarp();
      if (MODE == 0) {
        // S^T of the first two steps, into tiles (gs) mod 2 and (gs + 1) mod 2
        for (int t = 0; ok && t < 2 && t < nt; ++t) {
          const uint32_t iq = i0 + 2 + 2 * t, b = (gs + t) & 1u;
          if (!(ok = wait(full + slot(iq), par(iq)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_st(iq, C::T_S + 64 * b);
            ptx::mma_commit(s_full + b);
            ptx::mma_commit(empty + slot(iq));   // Q is read by nothing later in this mode
          }
          __syncwarp();
        }
        for (int t = 0; ok && t < nt; ++t, ++gs) {
          const uint32_t b = gs & 1u, ph = (gs >> 1) & 1u;
          const uint32_t ido = i0 + 3 + 2 * t;
          // dV += P^T dO: P^T packed over S^T tile b (group g at columns [32g, 32g + 16)); the
          // unit's first product overwrites the accumulator, once the previous unit's is read out
          if (t == 0 && !(ok = wait(acc_free, (u_it & 1u) ^ 1u))) break;
          if (!(ok = wait(p_full + b, ph))) break;
          if (!(ok = wait(full + slot(ido), par(ido)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
#pragma unroll
            for (int kk = 0; kk < NS / 16; ++kk)
              ptx::mma_ts(tmem + C::T_ACC, tmem + C::T_S + 64 * b + 32 * (kk >> 1) + 8 * (kk & 1),
                          mnmaj64(aR + slot(ido) * SLOT, kk), C::IDESC_ACC, (t > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(empty + slot(ido));
          }
          __syncwarp();
          if (t + 2 < nt) {
            // S^T of step t + 2 into tile b, after the dV product that reads P^T from it
            const uint32_t iq = i0 + 2 + 2 * (t + 2);
            if (!(ok = wait(full + slot(iq), par(iq)))) break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
              moved |= lane != 0;
              mma_st(iq, C::T_S + 64 * b);
              ptx::mma_commit(s_full + b);
              ptx::mma_commit(empty + slot(iq));
            }
            __syncwarp();
          }
        }
      } else {
        if (!(ok = wait(v_full, u_it & 1u))) break;
        auto mma_dpt = [&](uint32_t ido) {   // dP^T = V dO^T: V resident (K-major over dv), the dO rows of ido
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            ptx::mma_ss(tmem + C::T_DP, kmaj(aV, BOX128, kk), kmaj(aR + slot(ido) * SLOT, BOX64, kk), C::IDESC_ST,
                        kk > 0);
          ptx::mma_commit(dp_full);
          ptx::mma_commit(empty + slot(ido));   // dO is read by nothing later in this mode
        };
        // S^T and dP^T of the first step
        if (!(ok = wait(full + slot(i0 + 2), par(i0 + 2)))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
          mma_st(i0 + 2, C::T_S);
          ptx::mma_commit(s_full);
        }
        __syncwarp();
        if (!(ok = wait(full + slot(i0 + 3), par(i0 + 3)))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
          mma_dpt(i0 + 3);
          if (nt == 1) ptx::mma_commit(v_empty);
        }
        __syncwarp();
        for (int t = 0; ok && t < nt; ++t, ++gs) {
          const uint32_t iq = i0 + 2 + 2 * t;   // Q_t; dO_{t+1} = iq + 3, Q_{t+1} = iq + 2
          if (t + 1 < nt) {
            // S^T of the next step once the row threads hold this one
            if (!(ok = wait(s_free, gs & 1u))) break;
            if (!(ok = wait(full + slot(iq + 2), par(iq + 2)))) break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
              moved |= lane != 0;
              mma_st(iq + 2, C::T_S);
              ptx::mma_commit(s_full);
            }
            __syncwarp();
          }
          // dK += dS^T Q: dS^T packed over dP^T (group g at columns [32g, 32g + 16)), Q MN-major;
          // the unit's first product overwrites the accumulator, once the previous unit's is read out
          if (t == 0 && !(ok = wait(acc_free, (u_it & 1u) ^ 1u))) break;
          if (!(ok = wait(ds_full, gs & 1u))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
#pragma unroll
            for (int kk = 0; kk < NS / 16; ++kk)
              ptx::mma_ts(tmem + C::T_ACC, tmem + C::T_DP + 32 * (kk >> 1) + 8 * (kk & 1),
                          mnmaj64(aR + slot(iq) * SLOT, kk), C::IDESC_ACC, (t > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(empty + slot(iq));
          }
          __syncwarp();
          if (t + 1 < nt) {
            // dP^T of the next step, into the tile the dK product has just read
            if (!(ok = wait(full + slot(iq + 3), par(iq + 3)))) break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
              moved |= lane != 0;
              mma_dpt(iq + 3);
              if (t + 2 == nt) ptx::mma_commit(v_empty);   // the unit's last read of V
            }
            __syncwarp();
          }
        }
      }
      if (!ok) break;
      if (ptx::elect_one()) {
        moved |= lane != 0;
        ptx::mma_commit(acc_full);
      }
      __syncwarp();
      item = i0 + 2 + 2 * nt;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ row groups (thread = key row)
    const int g = (warp - 2) >> 2;          // query columns [32g, 32g + 32) of each step
    const int quad = warp & 3;
    const int r = quad * 32 + lane;         // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tK = tmem + lane_off + C::T_K + 64 * g;
    const uint32_t tS = tmem + lane_off + C::T_S + 32 * g, tDP = tmem + lane_off + C::T_DP + 32 * g;
    const uint32_t tACC = tmem + lane_off + C::T_ACC;
    ptx::WaitCtx w{abort_flag, P.status, 23u + g};
    const float sc2 = P.sc2, scale = P.p.scale;
    uint32_t item = 0, u_it = 0, gs = 0, n = 0;
    bool ok = true;
    int bh, kb;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &kb); ++round) {
      int t0, nt;
      kv_steps(P, kb, &t0, &nt);
      const int key = kb * BT + r;
      const bool key_ok = key < Tk;
      constexpr int WACC = MODE == 0 ? DV : HD;
      __nv_bfloat16* orow = (MODE == 0 ? P.dV : P.dK) + (static_cast<size_t>(bh) * Tk + (key_ok ? key : 0)) * WACC;
      if (nt == 0) {
        // no query row sees this key tile: its gradient rows are zero
        if (key_ok)
          for (int c = g; c < WACC / 8; c += 2) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint32_t i0 = item;
      // stage this group's half of K row r (d columns [128g, 128g + 128)) into TMEM
      for (int h = 0; h < 2; ++h)
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(full + slot(i0 + h), par(i0 + h), w)))) break;
      if (!ok) break;
      {
        const uint8_t* sk = ring + slot(i0 + (r >> 6)) * SLOT;
        const int rl = r & 63;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 x = *reinterpret_cast<const uint4*>(sk + bwd::sw128_offset64(rl, 128 * g + 64 * half + 8 * k));
            v[4 * k] = x.x;
            v[4 * k + 1] = x.y;
            v[4 * k + 2] = x.z;
            v[4 * k + 3] = x.w;
          }
          ptx::tmem_st32(tK + 32 * half, v);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(k_ready);
      for (int t = 0; t < nt; ++t, ++gs, ++n) {
        const int qb = (t0 + t) * NS + 32 * g;   // query of this thread's first column
        const int ls = lslot(n);
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(l_full + ls, lpar(n), w)))) break;
        const float* nl = sL + ls * 2 * NS + 32 * g;
        const uint32_t b = MODE == 0 ? (gs & 1u) : 0u, ph = MODE == 0 ? ((gs >> 1) & 1u) : (gs & 1u);
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(s_full + b, ph, w)))) break;
        ptx::tc_fence_after();
        float p[32];
        {
          uint32_t v[32];
          ptx::tmem_ld32(tS + 64 * b, v);
          ptx::tmem_ld_wait(v);
          if (MODE == 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(s_free);
          }
          // P^T_{key, q} = 2^(s * scale * log2 e - LSE_q * log2 e): zero for a
          // key past Tk, a query before the key (causal) or a query row past
          // Tq (its -LSE*log2(e) is -inf)
          const int lim = !key_ok ? 32 : (P.p.causal ? key - qb : 0);   // columns [0, lim) masked
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 l4 = ptx::lds128(nl + i);
            const float2 x01 = ptx::ffma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                          make_float2(sc2, sc2), make_float2(l4.x, l4.y));
            const float2 x23 = ptx::ffma2(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])),
                                          make_float2(sc2, sc2), make_float2(l4.z, l4.w));
            p[i] = i < lim ? 0.f : ptx::ex2(x01.x);
            p[i + 1] = i + 1 < lim ? 0.f : ptx::ex2(x01.y);
            p[i + 2] = i + 2 < lim ? 0.f : ptx::ex2(x23.x);
            p[i + 3] = i + 3 < lim ? 0.f : ptx::ex2(x23.y);
          }
        }
        if (MODE == 0) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16(p[2 * i], p[2 * i + 1]);
          ptx::tmem_st16(tS + 64 * b, pk);   // over this group's own first 16 columns (already read)
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          ptx::mbar_arrive(p_full + b);
          ptx::mbar_arrive(l_empty + ls);
        } else {
          const float* dd = nl + NS;   // D of these queries
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dp_full, gs & 1u, w)))) break;
          ptx::tc_fence_after();
          uint32_t v[32];
          ptx::tmem_ld32(tDP, v);
          ptx::tmem_ld_wait(v);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 d4 = ptx::lds128(dd + i);
            const float2 e01 = ptx::fadd2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                          make_float2(-d4.x, -d4.y));
            const float2 e23 = ptx::fadd2(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])),
                                          make_float2(-d4.z, -d4.w));
            const float2 s01 = ptx::fmul2(make_float2(p[i], p[i + 1]), e01);
            const float2 s23 = ptx::fmul2(make_float2(p[i + 2], p[i + 3]), e23);
            pk[i / 2] = ptx::pack_bf16(s01.x, s01.y);
            pk[i / 2 + 1] = ptx::pack_bf16(s23.x, s23.y);
          }
          ptx::tmem_st16(tDP, pk);   // over this group's own first 16 columns of dP^T (already read)
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          ptx::mbar_arrive(ds_full);
          ptx::mbar_arrive(l_empty + ls);
        }
      }
      if (!ok) break;
      // epilogue: this group writes accumulator columns [g WACC / 2, (g + 1) WACC / 2) of key row r
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(acc_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      const float mul = MODE == 1 ? scale : 1.0f;   // dK = scale * dS^T Q
#pragma unroll 1
      for (int c = 0; c < WACC / 64; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(tACC + (WACC / 2) * g + 32 * c, v);
        ptx::tmem_ld_wait(v);
        if (key_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + (WACC / 2) * g + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(ptx::pack_bf16(__uint_as_float(v[8 * e]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
                                ptx::pack_bf16(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
                                ptx::pack_bf16(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
                                ptx::pack_bf16(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(acc_free);
      item = i0 + 2 + 2 * nt;
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

// --------------------------------------------------------------------------
// Query-tile kernel: dQ.

template <int DV>
struct CfgQ {
  static constexpr int DORES = BT * DV * 2;   // dO of the unit (A operand of dP), 128-row boxes
  static constexpr int DPART_BYTES = 2 * 2 * BT * 4;   // [unit parity][row group][128] fp32 partial D
  static constexpr int NSLOT_FIT = (227 * 1024 - DORES - DPART_BYTES - 512) / SLOT;
  static constexpr int NSLOT = NSLOT_FIT < 16 ? NSLOT_FIT : 16;
  static constexpr int OFF_DO = 0;
  static constexpr int OFF_RING = OFF_DO + DORES;
  static constexpr int OFF_DPART = OFF_RING + NSLOT * SLOT;
  static constexpr int OFF_BAR = OFF_DPART + DPART_BYTES;
  // full[NSLOT], empty[NSLOT], q_ready, do_full, do_empty, s_full, s_free, dp_full, ds_full, dq_full,
  // dq_free, drain, dpart_full
  static constexpr int NBAR = 2 * NSLOT + 11;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16(BT, NS, false, false);   // S, dP: N = 64 keys
  static constexpr uint32_t IDESC_DQ = ptx::idesc_bf16(BT, HD, false, true);   // dQ: N = 256, K MN-major
  static constexpr uint32_t T_Q = 0, T_S = 128, T_DP = 192, T_DQ = 256;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NSLOT >= 4, "ring");
};

// Key steps of query tile qt: the 64-key steps below Tk and, causal, below
// the end of the tile.
__device__ __forceinline__ int q_steps(const Params& P, int qt) {
  int end = (P.p.Tk + NS - 1) / NS;
  if (P.p.causal) end = min(end, 2 * (qt + 1));
  return end;
}

template <int DV>
__global__ void __launch_bounds__(THREADS, 1)
    q256_kernel(const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ CUtensorMap tmK64,
                const __grid_constant__ CUtensorMap tmV64, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmO64, const Params P) {
  using C = CfgQ<DV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(P.status, ATTN_DEV_BAD_SMEM);
    return;
  }
  uint8_t* sdO = smem + C::OFF_DO;
  uint8_t* ring = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = full + C::NSLOT;
  uint64_t* q_ready = empty + C::NSLOT;   // the row threads staged the unit's Q into TMEM
  uint64_t* do_full = q_ready + 1;
  uint64_t* do_empty = q_ready + 2;
  uint64_t* s_full = q_ready + 3;
  uint64_t* s_free = q_ready + 4;
  uint64_t* dp_full = q_ready + 5;
  uint64_t* ds_full = q_ready + 6;
  uint64_t* dq_full = q_ready + 7;
  uint64_t* dq_free = q_ready + 8;        // the epilogue has read the dQ accumulator
  uint64_t* drain = q_ready + 9;
  uint64_t* dpart_full = q_ready + 10;    // both row groups wrote a unit's partial D
  float* dpart = reinterpret_cast<float*>(smem + C::OFF_DPART);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(full + s, 1);
      ptx::mbar_init(empty + s, 1);
    }
    ptx::mbar_init(q_ready, 256);
    ptx::mbar_init(do_full, 1);
    // the unit's last dP product has read dO, and the row threads have formed D from it
    ptx::mbar_init(do_empty, 2);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_free, 256);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(ds_full, 256);
    ptx::mbar_init(dq_full, 1);
    ptx::mbar_init(dq_free, 256);
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
  const int grid = gridDim.x, cta = blockIdx.x;
  const int Tq = P.p.Tq, Tk = P.p.Tk;
  // Ring items: per unit the halves of its Q tile at i0, i0 + 1 and of its O
  // tile at i0 + 2, i0 + 3, then per key step s the 64 rows of K at
  // i0 + 4 + 2s and of V at i0 + 5 + 2s.
  auto slot = [](uint32_t i) { return static_cast<int>(i % C::NSLOT); };
  auto par = [](uint32_t i) { return (i / C::NSLOT) & 1u; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::WaitCtx w{abort_flag, P.status, 25u};
    ptx::tma_prefetch_desc(&tmQ64);
    ptx::tma_prefetch_desc(&tmK64);
    ptx::tma_prefetch_desc(&tmV64);
    ptx::tma_prefetch_desc(&tmdO);
    ptx::tma_prefetch_desc(&tmO64);
    uint32_t item = 0, u_it = 0, d_issued = 0;
    bool ok = true;
    int bh, qt;
    auto load = [&](const CUtensorMap* map, int boxes, uint32_t bytes, int row) {
      const int s = slot(item);
      if (!ptx::mbar_wait(empty + s, par(item) ^ 1u, w)) return false;
      ptx::mbar_arrive_expect_tx(full + s, bytes);
      for (int b = 0; b < boxes; ++b) ptx::tma_load_3d(ring + s * SLOT + b * BOX64, map, full + s, b * 64, row, bh);
      ++item;
      return true;
    };
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &qt); ++round) {
      const int ns = q_steps(P, qt);
      if (ns == 0) continue;
      ok = load(&tmQ64, HD / 64, 64 * HD * 2, qt * BT) && load(&tmQ64, HD / 64, 64 * HD * 2, qt * BT + 64) &&
           load(&tmO64, DV / 64, 64 * DV * 2, qt * BT) && load(&tmO64, DV / 64, 64 * DV * 2, qt * BT + 64);
      if (!ok) break;
      // dO of the unit, once the previous unit's last dP product and D have read it
      if (!(ok = ptx::mbar_wait(do_empty, (u_it & 1u) ^ 1u, w))) break;
      ptx::mbar_arrive_expect_tx(do_full, BT * DV * 2);
      for (int b = 0; b < DV / 64; ++b) ptx::tma_load_3d(sdO + b * BOX128, &tmdO, do_full, b * 64, qt * BT, bh);
      d_issued = u_it + 1;
      for (int s = 0; ok && s < ns; ++s)
        ok = load(&tmK64, HD / 64, 64 * HD * 2, s * NS) && load(&tmV64, DV / 64, 64 * DV * 2, s * NS);
      ++u_it;
    }
    if (!ok) {
      for (uint32_t m = (item > static_cast<uint32_t>(C::NSLOT) ? item - C::NSLOT : 0u); m < item; ++m)
        ptx::mbar_wait_drain(full + slot(m), par(m));
      if (d_issued > 0) ptx::mbar_wait_drain(do_full, (d_issued - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    ptx::WaitCtx w{abort_flag, P.status, 26u};
    const uint32_t aR = ptx::smem_u32(ring), adO = ptx::smem_u32(sdO);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, w));
    };
    auto mma_s = [&](uint32_t ik) {   // S = Q K^T: Q from TMEM, the K rows of item ik
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        ptx::mma_ts(tmem + C::T_S, tmem + C::T_Q + 8 * kk, kmaj(aR + slot(ik) * SLOT, BOX64, kk), C::IDESC_S, kk > 0);
      ptx::mma_commit(s_full);
    };
    auto mma_dp = [&](uint32_t iv, bool last) {   // dP = dO V^T: dO resident, the V rows of item iv
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk)
        ptx::mma_ss(tmem + C::T_DP, kmaj(adO, BOX128, kk), kmaj(aR + slot(iv) * SLOT, BOX64, kk), C::IDESC_S,
                    kk > 0);
      ptx::mma_commit(dp_full);
      ptx::mma_commit(empty + slot(iv));
      if (last) ptx::mma_commit(do_empty);   // the unit's last read of dO
    };
    uint32_t item = 0, u_it = 0, gs = 0;
    bool ok = true, moved = false;
    int bh, qt;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &qt); ++round) {
      const int ns = q_steps(P, qt);
      if (ns == 0) continue;
      const uint32_t i0 = item;
      if (!(ok = wait(q_ready, u_it & 1u))) break;
      if (lane == 0) {
        ptx::mbar_arrive(empty + slot(i0));
        ptx::mbar_arrive(empty + slot(i0 + 1));
      }
      __syncwarp();
      if (!(ok = wait(full + slot(i0 + 4), par(i0 + 4)))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        mma_s(i0 + 4);
      }
      __syncwarp();
      if (!(ok = wait(do_full, u_it & 1u))) break;
      if (!(ok = wait(full + slot(i0 + 5), par(i0 + 5)))) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        moved |= lane != 0;
        mma_dp(i0 + 5, ns == 1);
      }
      __syncwarp();
      for (int s = 0; ok && s < ns; ++s, ++gs) {
        const uint32_t ik = i0 + 4 + 2 * s;   // K_s; K_{s+1} = ik + 2, V_{s+1} = ik + 3
        if (s + 1 < ns) {
          if (!(ok = wait(s_free, gs & 1u))) break;
          if (!(ok = wait(full + slot(ik + 2), par(ik + 2)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_s(ik + 2);
          }
          __syncwarp();
        }
        // dQ += dS K: dS packed over dP (group g at columns [32g, 32g + 16)), K MN-major; the
        // unit's first product overwrites the accumulator, once the previous unit's is read out
        if (s == 0 && !(ok = wait(dq_free, (u_it & 1u) ^ 1u))) break;
        if (!(ok = wait(ds_full, gs & 1u))) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          moved |= lane != 0;
#pragma unroll
          for (int kk = 0; kk < NS / 16; ++kk)
            ptx::mma_ts(tmem + C::T_DQ, tmem + C::T_DP + 32 * (kk >> 1) + 8 * (kk & 1),
                        mnmaj64(aR + slot(ik) * SLOT, kk), C::IDESC_DQ, (s > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(empty + slot(ik));
        }
        __syncwarp();
        if (s + 1 < ns) {
          if (!(ok = wait(full + slot(ik + 3), par(ik + 3)))) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            moved |= lane != 0;
            mma_dp(ik + 3, s + 2 == ns);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (ptx::elect_one()) {
        moved |= lane != 0;
        ptx::mma_commit(dq_full);
      }
      __syncwarp();
      item = i0 + 4 + 2 * ns;
      ++u_it;
    }
    if (!ok) {
      if (ptx::elect_one()) ptx::mma_commit(drain);
      __syncwarp();
      ptx::mbar_wait_drain(drain, 0u);
    }
    if (__any_sync(0xffffffffu, moved) && lane == 0) atomicOr(P.status, ATTN_DEV_ISSUER);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ row groups (thread = query row)
    const int g = (warp - 2) >> 2;          // key columns [32g, 32g + 32) of each step
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tQ = tmem + lane_off + C::T_Q + 64 * g;
    const uint32_t tS = tmem + lane_off + C::T_S + 32 * g, tDP = tmem + lane_off + C::T_DP + 32 * g;
    const uint32_t tDQ = tmem + lane_off + C::T_DQ + 128 * g;
    ptx::WaitCtx w{abort_flag, P.status, 27u + g};
    const float sc2 = P.sc2, scale = P.p.scale;
    uint32_t item = 0, u_it = 0, gs = 0;
    bool ok = true;
    int bh, qt;
    for (int round = 0; ok && P.order.unit(cta, grid, round, &bh, &qt); ++round) {
      const int ns = q_steps(P, qt);
      if (ns == 0) continue;
      const uint32_t i0 = item;
      const int q = qt * BT + r;
      const bool q_ok = q < Tq;
      // -LSE*log2(e) of this row (-inf past Tq and for rows without keys)
      const float lse = q_ok ? P.LSE[static_cast<size_t>(bh) * Tq + q] : -CUDART_INF_F;
      const float nlse2 = lse == -CUDART_INF_F ? -CUDART_INF_F : -lse * LOG2E;
      // stage this group's half of Q row r (d columns [128g, 128g + 128)) into TMEM
      for (int h = 0; h < 2; ++h)
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(full + slot(i0 + h), par(i0 + h), w)))) break;
      if (!ok) break;
      {
        const uint8_t* sq = ring + slot(i0 + (r >> 6)) * SLOT;
        const int rl = r & 63;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 x = *reinterpret_cast<const uint4*>(sq + bwd::sw128_offset64(rl, 128 * g + 64 * half + 8 * k));
            v[4 * k] = x.x;
            v[4 * k + 1] = x.y;
            v[4 * k + 2] = x.z;
            v[4 * k + 3] = x.w;
          }
          ptx::tmem_st32(tQ + 32 * half, v);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(q_ready);
      // D = rowsum(dO o O) of this row ("attention_backprop", section
      // "Gradient of S"): this group's half of the dv columns from the
      // resident dO and the unit's O items, the two halves added through
      // shared memory (rows past Tq load as zeros, so their D is 0). Group 0
      // stores D and -LSE*log2(e) into the padded arrays the dV and dK
      // kernels read after this kernel.
      float dd;
      {
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(do_full, u_it & 1u, w)))) break;
        for (int h = 0; h < 2; ++h)
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(full + slot(i0 + 2 + h), par(i0 + 2 + h), w)))) break;
        if (!ok) break;
        const uint8_t* so = ring + slot(i0 + 2 + (r >> 6)) * SLOT;
        const int rl = r & 63;
        float part = 0.f;
#pragma unroll
        for (int k = 0; k < DV / 16; ++k) {
          const int c = (DV / 2) * g + 8 * k;
          const uint4 x = *reinterpret_cast<const uint4*>(sdO + bwd::sw128_offset(r, c));
          const uint4 o = *reinterpret_cast<const uint4*>(so + bwd::sw128_offset64(rl, c));
          const __nv_bfloat162* dv2 = reinterpret_cast<const __nv_bfloat162*>(&x);
          const __nv_bfloat162* ov2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = __bfloat1622float2(ov2[e]), b = __bfloat1622float2(dv2[e]);
            part = fmaf(a.x, b.x, part);
            part = fmaf(a.y, b.y, part);
          }
        }
        float* dpu = dpart + (u_it & 1u) * 2 * BT;
        dpu[g * BT + r] = part;
        ptx::mbar_arrive(dpart_full);
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dpart_full, u_it & 1u, w)))) break;
        dd = dpu[r] + dpu[BT + r];
        if (g == 0) {   // every row of the padded tile: the dV and dK kernels read whole slices
          P.D[static_cast<size_t>(bh) * P.Tq_pad + q] = dd;
          P.NLSE2[static_cast<size_t>(bh) * P.Tq_pad + q] = nlse2;
        }
        if (threadIdx.x == 64) {
          // every row thread has read the O items and dO for D
          ptx::mbar_arrive(empty + slot(i0 + 2));
          ptx::mbar_arrive(empty + slot(i0 + 3));
          ptx::mbar_arrive(do_empty);
        }
      }
      for (int s = 0; s < ns; ++s, ++gs) {
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(s_full, gs & 1u, w)))) break;
        ptx::tc_fence_after();
        float p[32];
        {
          uint32_t v[32];
          ptx::tmem_ld32(tS, v);
          ptx::tmem_ld_wait(v);
          ptx::tc_fence_before();
          ptx::mbar_arrive(s_free);
          const int kv0 = s * NS + 32 * g;   // key of this thread's first column
          // keys [lim, 32) of this thread's columns are past Tk or (causal) after the query
          const int lim = min(Tk - kv0, P.p.causal ? q - kv0 + 1 : 32);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = ptx::ffma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                        make_float2(sc2, sc2), make_float2(nlse2, nlse2));
            p[i] = i < lim ? ptx::ex2(x.x) : 0.f;
            p[i + 1] = i + 1 < lim ? ptx::ex2(x.y) : 0.f;
          }
        }
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dp_full, gs & 1u, w)))) break;
        ptx::tc_fence_after();
        uint32_t v[32];
        ptx::tmem_ld32(tDP, v);
        ptx::tmem_ld_wait(v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 e = ptx::fadd2(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                      make_float2(-dd, -dd));
          const float2 rr = ptx::fmul2(make_float2(p[2 * i], p[2 * i + 1]), e);
          pk[i] = ptx::pack_bf16(rr.x, rr.y);
        }
        ptx::tmem_st16(tDP, pk);   // over this group's own first 16 columns of dP (already read)
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ds_full);
      }
      if (!ok) break;
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(dq_full, u_it & 1u, w)))) break;
      ptx::tc_fence_after();
      // this group writes dQ columns [128g, 128g + 128) of its row
      __nv_bfloat16* row = P.dQ + (static_cast<size_t>(bh) * Tq + (q_ok ? q : 0)) * HD + 128 * g;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(tDQ + 32 * c, v);
        ptx::tmem_ld_wait(v);
        if (q_ok) {
          uint4* dst = reinterpret_cast<uint4*>(row + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                ptx::pack_bf16(__uint_as_float(v[8 * e]) * scale, __uint_as_float(v[8 * e + 1]) * scale),
                ptx::pack_bf16(__uint_as_float(v[8 * e + 2]) * scale, __uint_as_float(v[8 * e + 3]) * scale),
                ptx::pack_bf16(__uint_as_float(v[8 * e + 4]) * scale, __uint_as_float(v[8 * e + 5]) * scale),
                ptx::pack_bf16(__uint_as_float(v[8 * e + 6]) * scale, __uint_as_float(v[8 * e + 7]) * scale));
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(dq_free);
      item = i0 + 4 + 2 * ns;
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

// --------------------------------------------------------------------------

template <typename K>
cudaError_t prep(K kern, int smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int DV>
cudaError_t launch_t(const LaunchBwd& a, Params P) {
  const int heads = a.p.B * a.p.H;
  cudaError_t e;
  const bool all = a.phase == 0 || a.phase == 2;
  // phase 5: the dQ kernel; phase 4: the dV and dK kernels
  if (all || a.phase == 5) {
    P.order = Order{P.n_q_tiles, heads, a.p.causal ? 1 : 0};
    const long long units = static_cast<long long>(P.n_q_tiles) * heads;
    const int grid = units < a.num_sms ? static_cast<int>(units) : a.num_sms;
    auto kq = q256_kernel<DV>;
    if ((e = prep(kq, CfgQ<DV>::SMEM)) != cudaSuccess) return e;
    kq<<<grid, THREADS, CfgQ<DV>::SMEM, a.stream>>>(*a.tmQ64, *a.tmK64, *a.tmV64, *a.tmdO, *a.tmO64, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (all || a.phase == 4) {
    P.order = Order{P.n_k_tiles, heads, a.p.causal ? 2 : 0};
    const long long units = static_cast<long long>(P.n_k_tiles) * heads;
    const int grid = units < a.num_sms ? static_cast<int>(units) : a.num_sms;
    auto kv = kv256_kernel<DV, 0>;
    auto kk = kv256_kernel<DV, 1>;
    if ((e = prep(kv, CfgKV<DV, 0>::SMEM)) != cudaSuccess) return e;
    if ((e = prep(kk, CfgKV<DV, 1>::SMEM)) != cudaSuccess) return e;
    kv<<<grid, THREADS, CfgKV<DV, 0>::SMEM, a.stream>>>(*a.tmQ64, *a.tmK64, *a.tmV, *a.tmdO64, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kk<<<grid, THREADS, CfgKV<DV, 1>::SMEM, a.stream>>>(*a.tmQ64, *a.tmK64, *a.tmV, *a.tmdO64, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bwd256

// The bf16 backward for d = 256 (dv 64, 128 or 256): the dQ kernel (phase 5),
// which also forms D and -LSE * log2(e), then the dV and dK kernels (phase 4);
// dQ is written directly (no conversion phase) and phase 1 launches nothing.
cudaError_t launch_bwd_bf16_d256(const LaunchBwd& a) {
  const Problem& p = a.p;
  bwd::Params P{};
  P.p = p;
  P.NLSE2 = a.NLSE2;
  P.D = a.D;
  P.LSE = a.LSE;
  P.Tq_pad = padded_rows(p.Tq);
  P.dQ = static_cast<__nv_bfloat16*>(a.dQ);
  P.dK = static_cast<__nv_bfloat16*>(a.dK);
  P.dV = static_cast<__nv_bfloat16*>(a.dV);
  P.status = a.status;
  P.n_q_tiles = (p.Tq + bwd::BT - 1) / bwd::BT;
  P.n_k_tiles = (p.Tk + bwd::BT - 1) / bwd::BT;
  P.sc2 = p.scale * bwd::LOG2E;
  if (static_cast<long long>(P.n_q_tiles) * p.B * p.H > 0x7fffffffLL ||
      static_cast<long long>(P.n_k_tiles) * p.B * p.H > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  if (p.dv == 256) return bwd256::launch_t<256>(a, P);
  if (p.dv == 128) return bwd256::launch_t<128>(a, P);
  return bwd256::launch_t<64>(a, P);
}

}  // namespace attn
