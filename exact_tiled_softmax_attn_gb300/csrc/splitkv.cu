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

// One warp per output row; lane c handles columns [4c, 4c + 4) and, for dv
// above 128, [128 + 4c, 128 + 4c + 4) (dv <= 256).
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
    // (the d <= 128 forward pairs query tiles as 2 qb, 2 qb + 1, the d = 256
    // one takes them singly; with 128-key tiles either way)
    const int qt = q / 128;
    const int nt = causal ? min(qt + 1, n_kv_tiles) : n_kv_tiles;
    const int ns = min(n_splits, (nt + split_tiles - 1) / split_tiles);
    // the loops over splits are unrolled so that several partial rows are in
    // flight at once (the kernel is bound by load latency, not bandwidth)
    float mx = -CUDART_INF_F;
#pragma unroll 4
    for (int s = 0; s < ns; ++s) mx = fmaxf(mx, LSEpart[static_cast<long long>(s) * rows + r]);
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    float lse = -CUDART_INF_F;
    if (mx != -CUDART_INF_F) {
      float wsum = 0.f;
#pragma unroll 4
      for (int s = 0; s < ns; ++s) {
        const float ls = LSEpart[static_cast<long long>(s) * rows + r];
        const float wgt = expf(ls - mx);   // 0 for a split with no allowed key
        wsum += wgt;
        const float4* orow = reinterpret_cast<const float4*>(Opart + (static_cast<long long>(s) * rows + r) * dv);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (4 * (lane + 32 * h) < dv) {
            const float4 o = orow[lane + 32 * h];
            acc[h].x = fmaf(wgt, o.x, acc[h].x);
            acc[h].y = fmaf(wgt, o.y, acc[h].y);
            acc[h].z = fmaf(wgt, o.z, acc[h].z);
            acc[h].w = fmaf(wgt, o.w, acc[h].w);
          }
        }
      }
      const float inv = 1.0f / wsum;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        acc[h].x *= inv;
        acc[h].y *= inv;
        acc[h].z *= inv;
        acc[h].w *= inv;
      }
      lse = mx + logf(wsum);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (4 * (lane + 32 * h) < dv) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[h].x, acc[h].y), hi = __floats2bfloat162_rn(acc[h].z, acc[h].w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(O + r * dv)[lane + 32 * h] = pk;
      }
    }
    if (lane == 0) LSE[r] = lse;
  }
}

// The same merge for fp32 outputs (the CUDA-core forward's key ranges): one
// warp per output row, lane c handling columns c, c + 32, ... (any dv up to
// 256, rows with no alignment beyond 4 bytes). The partial log-sum-exps are
// fp64: at logits in the thousands an fp32 LSE_s is off by up to 1e-4. Lane
// s holds split s's (and split s + 32's): the maximum M is taken over the
// warp in fp64 and each weight exp(LSE_s - M) from the fp64 difference
// rounded to fp32, whose error (|LSE_s - M| * 2^-24) matters only where the
// weight does not vanish. The weights and their sum are fp32 from there on,
// and every lane forms the same sum (a butterfly of commutative adds).
// `tile`: rows per query tile and keys per key tile of the forward that
// wrote the partials.
__global__ void __launch_bounds__(NT) merge_f32_kernel(const float* __restrict__ Opart,
                                                       const double* __restrict__ LSEpart, float* __restrict__ O,
                                                       float* __restrict__ LSE, long long rows, int Tq, int dv,
                                                       int n_splits, int split_tiles, int n_kv_tiles, int tile,
                                                       int causal) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * NT + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * NT) >> 5;
  for (long long r = warp_id; r < rows; r += n_warps) {
    const int q = static_cast<int>(r % Tq);
    // the ranges the forward ran for this row's query tile (key tiles up to
    // the diagonal tile under the causal mask)
    const int qt = q / tile;
    const int nt = causal ? min(qt + 1, n_kv_tiles) : n_kv_tiles;
    const int ns = min(n_splits, (nt + split_tiles - 1) / split_tiles);   // <= 64
    const double l0 = lane < ns ? LSEpart[static_cast<long long>(lane) * rows + r] : -CUDART_INF;
    const double l1 = lane + 32 < ns ? LSEpart[static_cast<long long>(lane + 32) * rows + r] : -CUDART_INF;
    double mx = fmax(l0, l1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = 0.f;
    float lse = -CUDART_INF_F;
    if (mx != -CUDART_INF) {
      // 0 for a split with no allowed key (LSE_s = -inf)
      const float w0 = expf(static_cast<float>(l0 - mx));
      const float w1 = expf(static_cast<float>(l1 - mx));
      float wsum = w0 + w1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
      for (int s = 0; s < ns; ++s) {
        const float wgt = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
        const float* orow = Opart + (static_cast<long long>(s) * rows + r) * dv;
#pragma unroll
        for (int h = 0; h < 8; ++h)
          if (lane + 32 * h < dv) acc[h] = fmaf(wgt, orow[lane + 32 * h], acc[h]);
      }
      const float inv = 1.0f / wsum;
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[h] *= inv;
      lse = static_cast<float>(mx + static_cast<double>(logf(wsum)));
    }
#pragma unroll
    for (int h = 0; h < 8; ++h)
      if (lane + 32 * h < dv) O[r * dv + lane + 32 * h] = acc[h];
    if (lane == 0) LSE[r] = lse;
  }
}

}  // namespace splitkv

cudaError_t launch_splitkv_merge_f32(const Problem& p, const float* Opart, const double* LSEpart, int n_splits,
                                     int split_tiles, int tile, float* O, float* LSE, int num_sms, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Tq;
  if (rows == 0) return cudaSuccess;
  if (p.dv > 256 || n_splits < 1 || n_splits > splitkv::kMaxSplits || split_tiles < 1 || tile < 1)
    return cudaErrorInvalidValue;
  const long long want = (rows + splitkv::NT / 32 - 1) / (splitkv::NT / 32);
  const int grid = static_cast<int>(want < num_sms * 16LL ? want : num_sms * 16LL);
  splitkv::merge_f32_kernel<<<grid, splitkv::NT, 0, s>>>(Opart, LSEpart, O, LSE, rows, p.Tq, p.dv, n_splits,
                                                         split_tiles, (p.Tk + tile - 1) / tile, tile, p.causal);
  return cudaGetLastError();
}

cudaError_t launch_splitkv_merge(const Problem& p, const float* Opart, const float* LSEpart, int n_splits,
                                 int split_tiles, void* O, float* LSE, int num_sms, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Tq;
  if (rows == 0) return cudaSuccess;
  if (p.dv > 256 || p.dv % 4 != 0 || n_splits < 1 || n_splits > splitkv::kMaxSplits || split_tiles < 1)
    return cudaErrorInvalidValue;
  const long long want = (rows + splitkv::NT / 32 - 1) / (splitkv::NT / 32);
  const int grid = static_cast<int>(want < num_sms * 16LL ? want : num_sms * 16LL);
  splitkv::merge_kernel<<<grid, splitkv::NT, 0, s>>>(Opart, LSEpart, static_cast<__nv_bfloat16*>(O), LSE, rows, p.Tq,
                                                     p.dv, n_splits, split_tiles, (p.Tk + 127) / 128, p.causal);
  return cudaGetLastError();
}

}  // namespace attn
