// Shared between the host layer (attn_api.cu) and the CUDA-core kernels
// (simt_f32.cu): the tiling the fp32 split-KV forward and split dQ count in.
#pragma once

namespace attn {

// Rows of the fp32 kernels' query tiles and keys of their key tiles when
// their keys are split into ranges (attn_fwd_splitkv, the split dQ).
constexpr int kF32SplitTile = 64;

}  // namespace attn
