// Memory-bound helper kernels: the backward preprocess D = rowsum(dO o O),
// the empty-key forward fill, and a zero fill.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace attn {
namespace small {

constexpr int NT = 256;

__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, const __nv_bfloat16*) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(x[i]);
    const float2 fy = __bfloat1622float2(y[i]);
    s = fmaf(fx.x, fy.x, s);
    s = fmaf(fx.y, fy.y, s);
  }
  return s;
}
__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, const float*) {
  const float* x = reinterpret_cast<const float*>(&a);
  const float* y = reinterpret_cast<const float*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) s = fmaf(x[i], y[i], s);
  return s;
}

// D_i = sum_c dO_ic * O_ic ("attention_backprop", section "Gradient of S":
// ROW_SUM(dL/dO o O); the delta-l term of "The Hidden Recurrence in Softmax
// Attention", section "Flash Attention Backward Pass"), written with the
// stored log-sum-exp in log2 units into [B*H, Tq_pad] arrays whose padding
// rows hold D = 0 and NLSE2 = -inf (so exp2(s + NLSE2) = 0 there). The backward
// fetches a 128-row slice of each with one bulk copy. Each group of LPR lanes
// reads a row with 16-byte loads, two rows at a time; rows are walked
// grid-stride. Optionally zeroes the matching row of an fp32 accumulator.
template <typename T>
__global__ void __launch_bounds__(NT) preprocess_vec(const T* __restrict__ O, const T* __restrict__ dO,
                                                      const float* __restrict__ LSE, float* __restrict__ D,
                                                      float* __restrict__ NLSE2, float* __restrict__ zero_rows,
                                                      int zero_cols, long long rows_pad, int Tq, int Tq_pad, int dv) {
  const int chunks = dv * static_cast<int>(sizeof(T)) / 16;   // 16-byte chunks per row (<= 32)
  const int lpr = chunks;                                      // lanes per row
  const int rows_per_warp = 32 / lpr;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lpr, c = lane - sub * lpr;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * NT + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * NT) >> 5;
  const long long step = n_warps * rows_per_warp;
  // two rows per lane group in flight: both rows' loads (O, dO chunks and
  // the LSE) are issued before either is reduced
  for (long long r0 = warp_id * rows_per_warp; r0 < rows_pad; r0 += 2 * step) {
    long long rp[2], r[2];
    bool inside[2], real[2];
    float lse[2], s[2];
    uint4 a[2], b[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rp[u] = r0 + u * step + sub;
      const long long bh = rp[u] / Tq_pad;
      const int q = static_cast<int>(rp[u] - bh * Tq_pad);
      r[u] = bh * Tq + q;                                      // unpadded row
      inside[u] = (sub < rows_per_warp) && (rp[u] < rows_pad);
      real[u] = inside[u] && q < Tq;
      lse[u] = (real[u] && c == 0) ? LSE[r[u]] : -CUDART_INF_F;
      if (real[u]) {
        a[u] = reinterpret_cast<const uint4*>(O + r[u] * dv)[c];
        b[u] = reinterpret_cast<const uint4*>(dO + r[u] * dv)[c];
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      s[u] = real[u] ? dot16(a[u], b[u], static_cast<const T*>(nullptr)) : 0.f;
      for (int o = lpr >> 1; o > 0; o >>= 1) s[u] += __shfl_xor_sync(0xffffffffu, s[u], o);
      if (inside[u] && c == 0) {
        D[rp[u]] = s[u];
        NLSE2[rp[u]] = (lse[u] == -CUDART_INF_F) ? -CUDART_INF_F : -lse[u] * 1.4426950408889634f;
      }
      if (real[u] && zero_rows) {
        float4* z = reinterpret_cast<float4*>(zero_rows + r[u] * zero_cols);
        for (int k = c; k < zero_cols / 4; k += lpr) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// Generic fp32 version (any dv): one warp per padded row.
__global__ void __launch_bounds__(NT) preprocess_f32(const float* __restrict__ O, const float* __restrict__ dO,
                                                      const float* __restrict__ LSE, float* __restrict__ D,
                                                      float* __restrict__ NLSE2, float* __restrict__ zero_rows,
                                                      int zero_cols, long long rows_pad, int Tq, int Tq_pad, int dv) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * NT + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * NT) >> 5;
  for (long long rp = warp_id; rp < rows_pad; rp += n_warps) {
    const long long bh = rp / Tq_pad;
    const int q = static_cast<int>(rp - bh * Tq_pad);
    const long long r = bh * Tq + q;
    const float lse = (q < Tq && lane == 0) ? LSE[r] : -CUDART_INF_F;   // with the row loads
    float s = 0.f;
    if (q < Tq)
      for (int c = lane; c < dv; c += 32) s = fmaf(O[r * dv + c], dO[r * dv + c], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      D[rp] = s;
      NLSE2[rp] = (lse == -CUDART_INF_F) ? -CUDART_INF_F : -lse * 1.4426950408889634f;
    }
    if (zero_rows && q < Tq)
      for (int c = lane; c < zero_cols; c += 32) zero_rows[r * zero_cols + c] = 0.f;
  }
}

__global__ void fill_empty_kernel(uint8_t* O, size_t o_bytes, float* LSE, size_t n_lse) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < o_bytes; i += stride) O[i] = 0;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_lse; i += stride)
    LSE[i] = -CUDART_INF_F;
}

__global__ void zero_kernel(uint8_t* p, size_t bytes) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < bytes; i += stride) p[i] = 0;
}

// Row width change of a [rows][w] bf16 array into [rows][wp] (pad: wp >= w,
// the new columns zero) or [rows][wp] into [rows][w] (crop: the first w
// columns), in 16-byte units: w8 = w / 8 and wp8 = wp / 8 units per row.
// One thread per 16-byte unit of the destination.
__global__ void pad_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long rows, int w8,
                                int wp8) {
  const long long n = rows * wp8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const long long r = i / wp8;
    const int c = static_cast<int>(i - r * wp8);
    dst[i] = c < w8 ? src[r * w8 + c] : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void crop_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long rows, int wp8,
                                 int w8) {
  const long long n = rows * w8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const long long r = i / w8;
    const int c = static_cast<int>(i - r * w8);
    dst[i] = src[r * wp8 + c];
  }
}

}  // namespace small

cudaError_t launch_bwd_preprocess(const Problem& p, const void* O, const void* dO, const float* LSE, int elem_bytes,
                                  float* D, float* NLSE2, float* zero_rows, int zero_cols, int num_sms,
                                  cudaStream_t s) {
  const int Tq_pad = padded_rows(p.Tq);
  const long long rows_pad = static_cast<long long>(p.B) * p.H * Tq_pad;
  if (rows_pad == 0) return cudaSuccess;
  const int grid = num_sms * 8;
  const int chunks = p.dv * elem_bytes / 16;
  const bool vec = (p.dv * elem_bytes) % 16 == 0 && chunks <= 32 && (chunks & (chunks - 1)) == 0 &&
                   (reinterpret_cast<uintptr_t>(O) % 16 == 0) && (reinterpret_cast<uintptr_t>(dO) % 16 == 0) &&
                   (zero_rows == nullptr || (zero_cols % 4 == 0 && reinterpret_cast<uintptr_t>(zero_rows) % 16 == 0));
  if (elem_bytes == 2) {
    small::preprocess_vec<__nv_bfloat16><<<grid, small::NT, 0, s>>>(
        static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, D, NLSE2, zero_rows,
        zero_cols, rows_pad, p.Tq, Tq_pad, p.dv);
  } else if (vec) {
    small::preprocess_vec<float><<<grid, small::NT, 0, s>>>(static_cast<const float*>(O),
                                                             static_cast<const float*>(dO), LSE, D, NLSE2,
                                                             zero_rows, zero_cols, rows_pad, p.Tq, Tq_pad, p.dv);
  } else {
    small::preprocess_f32<<<grid, small::NT, 0, s>>>(static_cast<const float*>(O), static_cast<const float*>(dO),
                                                      LSE, D, NLSE2, zero_rows, zero_cols, rows_pad, p.Tq, Tq_pad,
                                                      p.dv);
  }
  return cudaGetLastError();
}

cudaError_t launch_fill_empty_fwd(const Problem& p, void* O, float* LSE, int elem_bytes, cudaStream_t s) {
  const size_t n_lse = static_cast<size_t>(p.B) * p.H * p.Tq;
  const size_t o_bytes = n_lse * p.dv * elem_bytes;
  if (n_lse == 0) return cudaSuccess;
  small::fill_empty_kernel<<<1024, 256, 0, s>>>(static_cast<uint8_t*>(O), o_bytes, LSE, n_lse);
  return cudaGetLastError();
}

cudaError_t launch_pad_rows(const void* src, void* dst, long long rows, int w, int wp, int num_sms,
                            cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (w % 8 || wp % 8 || w <= 0 || wp < w) return cudaErrorInvalidValue;
  small::pad_rows_kernel<<<num_sms * 8, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), rows,
                                                       w / 8, wp / 8);
  return cudaGetLastError();
}

cudaError_t launch_crop_rows(const void* src, void* dst, long long rows, int wp, int w, int num_sms,
                             cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (w % 8 || wp % 8 || w <= 0 || wp < w) return cudaErrorInvalidValue;
  small::crop_rows_kernel<<<num_sms * 8, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                        rows, wp / 8, w / 8);
  return cudaGetLastError();
}

cudaError_t launch_zero(void* ptr, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  small::zero_kernel<<<1024, 256, 0, s>>>(static_cast<uint8_t*>(ptr), bytes);
  return cudaGetLastError();
}

}  // namespace attn
