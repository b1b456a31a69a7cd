// Shared between the host layer (attn_api.cu) and the CUDA-core kernels
// (simt_f32.cu): the tiling the fp32 split-KV forward and split dQ count in.
#pragma once

namespace attn {

// Rows of the fp32 kernels' query tiles and keys of their key tiles when
// their keys are split into ranges (attn_fwd_splitkv, the split dQ).
constexpr int kF32SplitTile = 64;

// fp32 deterministic backward: with at most kF32FusedDqMaxBytes of partials
// (one [B,H,Tq,d] fp32 array per 64-key tile) the dK/dV kernel also forms
// each key tile's dQ share and writes it to the tile's own partial array (or,
// with one key tile, to dQ itself); the partials are then added in key-tile
// order, and no separate dQ kernel runs.
constexpr unsigned long long kF32FusedDqMaxBytes = 1ull << 30;
inline bool f32_fused_dq(int B, int H, int Tq, int Tk, int d) {
  const long long n = (Tk + kF32SplitTile - 1) / kF32SplitTile;
  if (n < 1) return false;
  const unsigned long long bytes = static_cast<unsigned long long>(n) * B * H * Tq * d * 4ull;
  return n == 1 || bytes <= kF32FusedDqMaxBytes;
}

}  // namespace attn
