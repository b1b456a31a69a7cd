// Definitions shared by the bf16 backward kernels (bwd_bf16.cu, dq_pair.cu):
// tile constants, the unit order, the kernel parameters, the deterministic dQ
// kernels' unit decoding, and the shared-memory and TMEM layouts of their
// operands.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

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
};

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
