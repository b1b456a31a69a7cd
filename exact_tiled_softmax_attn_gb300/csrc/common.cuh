// Shared definitions of the CUDA path: problem descriptor, device status
// codes, the persistent work order, and the launch helpers' signatures.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Device status word bits (OR-ed by kernels; read back by the host).
constexpr uint32_t ATTN_DEV_TIMEOUT = 1u;     // a bounded pipeline wait gave up
constexpr uint32_t ATTN_DEV_BAD_SMEM = 2u;    // dynamic shared memory not 1024-byte aligned
constexpr uint32_t ATTN_DEV_ISSUER = 4u;      // elect.sync picked a lane other than 0 to issue MMAs

// Upper bound on any single wait inside a kernel. Legitimate waits here last
// micro- to milliseconds; reaching this means a producer never arrived.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// One attention problem: tensors [B, H, T, d] contiguous, LSE [B, H, Tq].
struct Problem {
  int B, H, Tq, Tk, d, dv;
  float scale;   // softmax scale applied to Q K^T
  int causal;    // 1: key j blocked for query i when j > i (global indices)
};

// Persistent, causal-aware order of work units. Units are (head bh, block
// index) pairs. Under the causal mask later blocks carry more work, so the
// order lists the heaviest blocks first (longest-processing-time first) and
// walks the grid in a serpentine so that each CTA's k-th unit alternates
// between the heavy and the light end of the remaining list.
struct UnitOrder {
  int n_blocks;   // blocks per head
  int n_heads;    // B * H
  int heavy_last; // 1: block index b carries more work when b is larger

  __host__ __device__ int count() const { return n_blocks * n_heads; }

  // k-th unit (k = round * grid + ...) of CTA `cta` out of `grid`.
  __device__ bool unit(int cta, int grid, int round, int* bh, int* blk) const {
    const int base = round * grid;
    const int x = base + ((round & 1) ? (grid - 1 - cta) : cta);
    if (base >= count()) return false;
    if (x >= count()) return false;
    if (heavy_last) {
      *blk = n_blocks - 1 - x / n_heads;
      *bh = x % n_heads;
    } else {
      *bh = x / n_blocks;
      *blk = x % n_blocks;
    }
    return true;
  }
};

}  // namespace attn
