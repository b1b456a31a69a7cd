// Merge of the split-KV forward's partial results.
//
// Split s of a query row holds the softmax over its own key range: O_s =
// A_s / l_s and LSE_s = m_s + log l_s. The whole row is the associative merge
// of the per-split states ("The Hidden Recurrence in Softmax Attention",
// section "Chunk-wise Mode with Online Softmax Re-scale": the running max, sum
// and accumulator of one key chunk rescaled to a common maximum and added):
//   M   = max_s LSE_s
//   w_s = exp(LSE_s - M),  W = sum_s w_s
//   O   = sum_s w_s O_s / W,  LSE = M + log W
// A split whose keys are all masked for the row has LSE_s = -inf and weight 0;
// a row with no allowed key at all gets O = 0, LSE = -inf.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace attn {
namespace splitkv {

constexpr int NT = 256;
constexpr int kMaxSplits = 64;

// One warp per output row; lane c handles columns [4c, 4c + 4) (dv <= 128).
__global__ void __launch_bounds__(NT) merge_kernel(const float* __restrict__ Opart, const float* __restrict__ LSEpart,
                                                   __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
                                                   long long rows, int Tq, int dv, int n_splits, int split_tiles,
                                                   int n_kv_tiles, int causal) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * NT + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * NT) >> 5;
  for (long long r = warp_id; r < rows; r += n_warps) {
    const int q = static_cast<int>(r % Tq);
    // key tiles of this row's query tile, as the forward's units count them
    // (query tiles pair up as 2 qb, 2 qb + 1)
    const int qt = q / 128;
    const int nt = causal ? min(qt + 1, n_kv_tiles) : n_kv_tiles;
    const int ns = min(n_splits, (nt + split_tiles - 1) / split_tiles);
    // the loops over splits are unrolled so that several partial rows are in
    // flight at once (the kernel is bound by load latency, not bandwidth)
    float mx = -CUDART_INF_F;
#pragma unroll 4
    for (int s = 0; s < ns; ++s) mx = fmaxf(mx, LSEpart[static_cast<long long>(s) * rows + r]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -CUDART_INF_F;
    if (mx != -CUDART_INF_F) {
      float wsum = 0.f;
#pragma unroll 4
      for (int s = 0; s < ns; ++s) {
        const float ls = LSEpart[static_cast<long long>(s) * rows + r];
        const float wgt = expf(ls - mx);   // 0 for a split with no allowed key
        wsum += wgt;
        if (4 * lane < dv) {
          const float4 o = reinterpret_cast<const float4*>(Opart + (static_cast<long long>(s) * rows + r) * dv)[lane];
          acc.x = fmaf(wgt, o.x, acc.x);
          acc.y = fmaf(wgt, o.y, acc.y);
          acc.z = fmaf(wgt, o.z, acc.z);
          acc.w = fmaf(wgt, o.w, acc.w);
        }
      }
      const float inv = 1.0f / wsum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      lse = mx + logf(wsum);
    }
    if (4 * lane < dv) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(O + r * dv)[lane] = pk;
    }
    if (lane == 0) LSE[r] = lse;
  }
}

}  // namespace splitkv

cudaError_t launch_splitkv_merge(const Problem& p, const float* Opart, const float* LSEpart, int n_splits,
                                 int split_tiles, void* O, float* LSE, int num_sms, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Tq;
  if (rows == 0) return cudaSuccess;
  if (p.dv > 128 || p.dv % 4 != 0 || n_splits < 1 || n_splits > splitkv::kMaxSplits || split_tiles < 1)
    return cudaErrorInvalidValue;
  const long long want = (rows + splitkv::NT / 32 - 1) / (splitkv::NT / 32);
  const int grid = static_cast<int>(want < num_sms * 16LL ? want : num_sms * 16LL);
  splitkv::merge_kernel<<<grid, splitkv::NT, 0, s>>>(Opart, LSEpart, static_cast<__nv_bfloat16*>(O), LSE, rows, p.Tq,
                                                     p.dv, n_splits, split_tiles, (p.Tk + 127) / 128, p.causal);
  return cudaGetLastError();
}

}  // namespace attn
