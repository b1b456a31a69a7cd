// One step of the online softmax on the device: fold one block of keys into
// the running (m, l, acc) state of every query row ("Tiled attention with an
// online softmax", section "Task"; the same recurrence as "The Hidden
// Recurrence in Softmax Attention", section "Chunk-wise Mode with Online
// Softmax Re-scale"). For row i and a block of bs scores s_ij with values v_j:
//   m' = max(m, max_j s_ij);  ref = (m' == -inf) ? 0 : m'   (the -inf rule)
//   c  = exp(m - ref);  p_j = exp(s_ij - ref)
//   l' = c l + sum_j p_j;  acc' = c acc + sum_j p_j v_j
// State and inputs are fp32; the arithmetic runs in fp64.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "launch.h"

namespace attn {
namespace step {

constexpr int NT = 128;       // threads per row
constexpr int CHUNK = 1024;   // scores of a row held in shared memory at a time

__global__ void __launch_bounds__(NT) online_softmax_step_kernel(float* __restrict__ m, float* __restrict__ l,
                                                                  float* __restrict__ acc,
                                                                  const float* __restrict__ scores,
                                                                  const float* __restrict__ v, int bs, int dv) {
  __shared__ double sp[CHUNK];
  __shared__ double red[NT / 32];
  const int row = blockIdx.x;
  const float* s = scores + static_cast<size_t>(row) * bs;
  // block maximum
  double bmax = -CUDART_INF;
  for (int j = threadIdx.x; j < bs; j += NT) bmax = fmax(bmax, static_cast<double>(s[j]));
  for (int o = 16; o > 0; o >>= 1) bmax = fmax(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = bmax;
  __syncthreads();
  bmax = red[0];
  for (int w = 1; w < NT / 32; ++w) bmax = fmax(bmax, red[w]);
  __syncthreads();
  const double m_old = m[row];
  const double m_new = fmax(m_old, bmax);
  const double ref = (m_new == -CUDART_INF) ? 0.0 : m_new;
  const double c = exp(m_old - ref);   // 0 when m_old = -inf
  // acc' = c acc + sum_j p_j v_j, one or more output columns per thread
  double lsum = 0.0;
  double a[4] = {0.0, 0.0, 0.0, 0.0};   // columns threadIdx.x + NT * k, k < 4 (dv <= 512)
  for (int j0 = 0; j0 < bs; j0 += CHUNK) {
    const int n = min(CHUNK, bs - j0);
    for (int j = threadIdx.x; j < n; j += NT) {
      const double p = exp(static_cast<double>(s[j0 + j]) - ref);   // 0 on blocked keys
      sp[j] = p;
      lsum += p;
    }
    __syncthreads();
    for (int j = 0; j < n; ++j) {
      const double p = sp[j];
      const float* vr = v + static_cast<size_t>(j0 + j) * dv;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int col = threadIdx.x + NT * k;
        if (col < dv) a[k] = fma(p, static_cast<double>(vr[col]), a[k]);
      }
    }
    __syncthreads();
  }
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lsum;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < NT / 32; ++w) t += red[w];
    m[row] = static_cast<float>(m_new);
    l[row] = static_cast<float>(c * static_cast<double>(l[row]) + t);
  }
  float* ar = acc + static_cast<size_t>(row) * dv;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int col = threadIdx.x + NT * k;
    if (col < dv) ar[col] = static_cast<float>(c * static_cast<double>(ar[col]) + a[k]);
  }
}

}  // namespace step

cudaError_t launch_online_softmax_step(float* m, float* l, float* acc, const float* scores, const float* v, int n,
                                       int bs, int dv, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  step::online_softmax_step_kernel<<<n, step::NT, 0, s>>>(m, l, acc, scores, v, bs, dv);
  return cudaGetLastError();
}

}  // namespace attn
