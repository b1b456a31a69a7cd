// Definitions shared by the bf16 backward kernels (bwd_bf16.cu, dq_pair.cu):
// tile constants, the unit order, the kernel parameters, the deterministic dQ
// kernels' unit decoding, and the shared-memory and TMEM layouts of their
// operands.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace bwd {

constexpr int BT = 128;                   // rows per tile (keys and queries)
constexpr int BOX_BYTES = 128 * 64 * 2;   // one TMA box: 128 rows x 64 bf16
constexpr float LOG2E = 1.4426950408889634f;

// Unit order: 0 = head-major, 1 = heavy (large block index) first,
// 2 = heavy (small block index) first.
struct Order {
  int n_blocks, n_heads, mode;
  __device__ bool unit(int cta, int grid, int round, int* bh, int* blk) const {
    const int base = round * grid;
    const int total = n_blocks * n_heads;
    if (base >= total) return false;
    const int x = base + ((round & 1) ? (grid - 1 - cta) : cta);
    if (x >= total) return false;
    if (mode == 0) {
      *bh = x / n_blocks;
      *blk = x % n_blocks;
    } else if (mode == 1) {
      *blk = n_blocks - 1 - x / n_heads;
      *bh = x % n_heads;
    } else {
      *blk = x / n_heads;
      *bh = x % n_heads;
    }
    return true;
  }
};

struct Params {
  Problem p;
  float* NLSE2;            // [BH, Tq_pad]: -LSE * log2(e), -inf on padding / no-key rows
  float* D;                // [BH, Tq_pad]
  const float* LSE;        // [BH, Tq] natural-log LSE from the forward
  int Tq_pad;
  float* dQacc;            // atomic path: fp32 [BH, Tq, d], pre-zeroed
  __nv_bfloat16* dQ;       // deterministic path output
  // deterministic dQ kernel split over key ranges (dq_splits > 1): split s of
  // a query tile covers key tiles [s * dq_split_tiles, (s + 1) * dq_split_tiles)
  // and writes scale * its partial dQ (fp32) to dQpart [dq_splits][BH*Tq][d];
  // a reduction adds the splits in order
  int dq_splits, dq_split_tiles;
  float* dQpart;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  uint32_t* status;
  Order order;
  int n_q_tiles, n_k_tiles;
  float sc2;               // scale * log2(e)
  // kernels whose producer hands units to the CTA's other roles (see
  // UnitQueue): dynamic = 1 claims them at run time from the launch's unit
  // counter `sched` (zeroed before the launch) in head groups of `group`;
  // dynamic = 0 takes the CTA's static share (every grid-th unit, serpentine)
  // of the same order with one group of all heads
  uint32_t* sched;
  int group;
  int dynamic;
};

// The r-th unit a CTA takes: claimed from the launch's counter (dynamic), or
// its static share of the sequence: unit r * grid + cta in even rounds and
// r * grid + grid - 1 - cta in odd ones, so that with the heaviest units
// first each CTA alternates between the heavy and the light end of what is
// left. Returns the unit count once the sequence is done.
__device__ __forceinline__ int next_unit_index(const Params& P, uint32_t r, int cta, int grid, int total) {
  if (P.dynamic) {
    const int x = static_cast<int>(atomicAdd(P.sched, 1u));
    return x < total ? x : total;
  }
  const long long base = static_cast<long long>(r) * grid;
  if (base >= total) return total;
  const long long x = base + ((r & 1u) ? grid - 1 - cta : cta);
  return x < total ? static_cast<int>(x) : total;
}

// Unit x (x < nb * nh) of a launch's sequence of units: heads in groups of
// `group`, the groups one after another, so that the operand tiles the
// units of a group share (K and V of a head for query-tile units, Q and dO
// for key-tile units) stay in L2 while the group runs; within a group the
// heaviest units first, the block index nb - 1 first when heavy_last and
// block 0 first otherwise (equal units in either order without a mask).
__device__ __forceinline__ void grouped_unit(int x, int nb, int nh, int group, bool heavy_last, int* bh, int* blk) {
  const int g = x / (nb * group);
  const int y = x - g * nb * group;
  const int hg = min(group, nh - g * group);
  const int b = y / hg;
  *blk = heavy_last ? nb - 1 - b : b;
  *bh = g * group + (y - b * hg);
}

// Units claimed at run time (Params::dynamic): the producer claims each unit
// with an atomic add on a global counter (next_unit_index), so a CTA that
// finishes early takes more units and the units of a head group run at about
// the same time, and publishes its index to the CTA's other roles through a
// ring of N slots in shared memory: slot u % N holds the CTA's u-th unit, or
// a value >= the unit count once the sequence is done. Every role reads every
// index in order (units without work included). With the static order each
// role computes the same sequence itself and the ring is not used.
struct UnitQueue {
  static constexpr int N = 4;
  volatile int* ids;   // [N] shared memory
  uint64_t* full;      // [N] arrived at by the producer when it wrote the slot
  uint64_t* empty;     // [N] arrived at once by each reader of the slot (count: all readers)
};

// Producer: publish x as the CTA's u-th unit (once every reader is done with
// the slot's previous index). False on a timeout.
__device__ __forceinline__ bool uq_push(const UnitQueue& q, uint32_t u, int x, const ptx::WaitCtx& w) {
  const int s = static_cast<int>(u % UnitQueue::N);
  if (!ptx::mbar_wait(q.empty + s, ((u / UnitQueue::N) & 1u) ^ 1u, w)) return false;
  q.ids[s] = x;
  ptx::mbar_arrive(q.full + s);   // (release: the index is seen by whoever acquires this phase)
  return true;
}

// Reader (every thread of the calling warp): the CTA's u-th unit index. The
// caller then arrives on q.empty[u % N] as its reader count says.
__device__ __forceinline__ bool uq_read(const UnitQueue& q, uint32_t u, int* x, const ptx::WaitCtx& w) {
  const int s = static_cast<int>(u % UnitQueue::N);
  if (!__all_sync(0xffffffffu, ptx::mbar_wait(q.full + s, (u / UnitQueue::N) & 1u, w))) return false;
  *x = q.ids[s];
  return true;
}


// Deterministic dQ unit `blk` of a head: query tile qt, key split s, first key
// tile j0 and key tile count nk (0 when the split lies past the tile's keys).
template <bool SPLIT>
__device__ __forceinline__ bool dq_unit(const Params& P, int blk, int* qt, int* s, int* j0, int* nk) {
  const int S = SPLIT ? P.dq_splits : 1;
  *qt = SPLIT ? blk / S : blk;
  *s = SPLIT ? blk - *qt * S : 0;
  const int n = P.p.causal ? min(*qt + 1, P.n_k_tiles) : P.n_k_tiles;
  *j0 = SPLIT ? *s * P.dq_split_tiles : 0;
  *nk = SPLIT ? max(0, min(n - *j0, P.dq_split_tiles)) : n;
  return *nk > 0;
}

// Byte offset of element (row, col) inside a 128-row tile stored as 64-column
// boxes with the 128-byte swizzle (the layout TMA writes and the MMA reads).
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  return (col >> 6) * BOX_BYTES + (row >> 3) * 1024 + (row & 7) * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
         (col & 7) * 2;
}

// Byte offset of element (row, col) of a 64-row tile stored as 64-column
// boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset64(int row, int col) {
  return (col >> 6) * (64 * 64 * 2) + (row >> 3) * 1024 + (row & 7) * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
         (col & 7) * 2;
}

// TMEM column of k-step kk (16 query columns, 8 packed columns) of the bf16
// P^T / dS^T operand: query columns 64h.. are packed at column 64h, where the
// half-h group read its fp32 scores, so no group overwrites columns the other
// group has not read yet.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

constexpr int DQ_PAIR_THREADS = 320;   // CTA-pair dQ kernel: producer, MMA, two row groups

// The deterministic dQ pass for d = 128 on CTA pairs (dq_pair.cu); P carries
// everything but the unit order, which it sets itself.
cudaError_t launch_dq_pair(const LaunchBwd& a, const Params& P);

}  // namespace bwd
}  // namespace attn
