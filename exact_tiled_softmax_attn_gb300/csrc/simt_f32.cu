// fp32 attention forward and backward on the CUDA cores.
//
// Same tiled algorithm as the tensor-core path ("Tiled attention with an
// online softmax", section "Task"; gradients from "attention_backprop",
// sections "Gradient of V and P", "Gradient of S", "Gradient of Q and K"),
// for fp32 inputs of any head size up to 256.
//
// Precision: a score q.k is accumulated in twice the fp32 precision (the
// compensated dot product below, fp32 instructions only) and held in fp64;
// scale * q.k and s - m are formed in fp64 before rounding to fp32 for exp.
// Accumulating s in plain fp32 instead leaves a logit error of ~1e-5..1e-4
// once |s| reaches the hundreds (keys scaled by +-40), which the softmax turns
// into output errors above 1e-5. Everything after the exponent (P, sums, P V,
// dP, dS, dQ, dK, dV) is fp32.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace attn {
namespace simt {

constexpr int BM = 32;          // query rows per tile
constexpr int NT = 256;         // threads per CTA
constexpr int MAXD = 256;       // largest supported d and dv

__device__ __forceinline__ double warp_max_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// sum_k a_k b_k by the compensated dot product of Ogita, Rump and Oishi
// ("Accurate Sum and Dot Product", SIAM J. Sci. Comput. 26(6), 2005,
// algorithm Dot2): each product splits exactly into p + e with one FMA, and
// the running sum is carried as s + c with Knuth's TwoSum, so the result is
// as accurate as a dot product accumulated in twice the fp32 precision while
// using only fp32 instructions (this GPU's fp64 rate is a small fraction of
// its fp32 rate). The _rn intrinsics keep the compiler from contracting the
// separate roundings the method relies on into FMAs. s + c is returned in
// fp64, where it is exact.
__device__ __forceinline__ double dot2(const float* a, const float* b, int n) {
  float s = 0.f, c = 0.f;
  for (int k = 0; k < n; ++k) {
    const float p = __fmul_rn(a[k], b[k]);
    const float e = __fmaf_rn(a[k], b[k], -p);   // a b - p, exactly
    const float t = __fadd_rn(s, p);
    const float z = __fsub_rn(t, s);
    const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(p, z));   // s + p - t, exactly
    s = t;
    c = __fadd_rn(c, __fadd_rn(err, e));
  }
  return static_cast<double>(s) + static_cast<double>(c);
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Copy `rows` x `cols` fp32 rows from global (row stride `cols`) into shared
// memory with row stride `ld`; rows at or beyond `valid` are zero.
__device__ __forceinline__ void load_rows(float* dst, int ld, const float* src, int rows, int cols, int valid) {
  for (int e = threadIdx.x; e < rows * cols; e += NT) {
    const int r = e / cols, c = e - r * cols;
    dst[r * ld + c] = (r < valid) ? src[static_cast<size_t>(r) * cols + c] : 0.f;
  }
}

// ---------------------------------------------------------------- forward

template <int BN>
__global__ void __launch_bounds__(NT) fwd_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                 const float* __restrict__ V, float* __restrict__ O,
                                                 float* __restrict__ LSE, const Problem p) {
  extern __shared__ double smem_d[];
  const int d = p.d, dv = p.dv, Tq = p.Tq, Tk = p.Tk;
  const int ldk = d + 1;
  double* sS = smem_d;                                  // [BM][BN+1]
  double* sM = sS + BM * (BN + 1);                      // [BM] running max (fp64, scaled logits)
  float* sQ = reinterpret_cast<float*>(sM + BM);        // [BM][d+1]
  float* sK = sQ + BM * ldk;                            // [BN][d+1]
  float* sV = sK + BN * ldk;                            // [BN][dv]
  float* sP = sV + BN * dv;                             // [BM][BN]
  float* sL = sP + BM * BN;                             // [BM] running sum
  float* sC = sL + BM;                                  // [BM] per-tile correction

  const int q0 = blockIdx.x * BM;
  const size_t bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const double scale = p.scale;

  load_rows(sQ, ldk, Q + (bh * Tq + q0) * d, BM, d, Tq - q0);
  if (threadIdx.x < BM) {
    sM[threadIdx.x] = -CUDART_INF;
    sL[threadIdx.x] = 0.f;
  }
  constexpr int PER = (BM * MAXD + NT - 1) / NT;   // O entries per thread
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;

  int n_kv = (Tk + BN - 1) / BN;
  if (p.causal) n_kv = min(n_kv, (q0 + BM - 1) / BN + 1);

  for (int jt = 0; jt < n_kv; ++jt) {
    const int kv0 = jt * BN;
    __syncthreads();
    load_rows(sK, ldk, K + (bh * Tk + kv0) * d, BN, d, Tk - kv0);
    load_rows(sV, dv, V + (bh * Tk + kv0) * dv, BN, dv, Tk - kv0);
    __syncthreads();
    // scores, compensated (twice fp32 precision) accumulation
    for (int e = threadIdx.x; e < BM * BN; e += NT) {
      const int i = e / BN, j = e - i * BN;
      const int qi = q0 + i, kj = kv0 + j;
      const double s = dot2(sQ + i * ldk, sK + j * ldk, d);
      const bool blocked = (kj >= Tk) || (p.causal && kj > qi);
      sS[i * (BN + 1) + j] = blocked ? -CUDART_INF : s * scale;
    }
    __syncthreads();
    // online softmax step, one warp per row
    for (int i = warp; i < BM; i += NT / 32) {
      double mx = -CUDART_INF;
      for (int j = lane; j < BN; j += 32) mx = fmax(mx, sS[i * (BN + 1) + j]);
      mx = warp_max_d(mx);
      const double m_old = sM[i];
      const double m_new = fmax(m_old, mx);
      const double ref = (m_new == -CUDART_INF) ? 0.0 : m_new;   // the -inf rule
      float sum = 0.f;
      for (int j = lane; j < BN; j += 32) {
        const float pj = expf(static_cast<float>(sS[i * (BN + 1) + j] - ref));
        sP[i * BN + j] = pj;
        sum += pj;
      }
      sum = warp_sum_f(sum);
      if (lane == 0) {
        const float corr = expf(static_cast<float>(m_old - ref));   // 0 when m_old = -inf
        sC[i] = corr;
        sL[i] = corr * sL[i] + sum;
        sM[i] = m_new;
      }
    }
    __syncthreads();
    // acc = corr * acc + P V
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = threadIdx.x + k * NT;
      if (e < BM * dv) {
        const int i = e / dv, c = e - i * dv;
        float a = acc[k] * sC[i];
        const float* pr = sP + i * BN;
        for (int j = 0; j < BN; ++j) a = fmaf(pr[j], sV[j * dv + c], a);
        acc[k] = a;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int e = threadIdx.x + k * NT;
    if (e < BM * dv) {
      const int i = e / dv, c = e - i * dv;
      if (q0 + i < Tq) {
        const float l = sL[i];
        O[(bh * Tq + q0 + i) * dv + c] = (l > 0.f) ? acc[k] / l : 0.f;
      }
    }
  }
  if (threadIdx.x < BM && q0 + threadIdx.x < Tq) {
    const int i = threadIdx.x;
    const float l = sL[i];
    LSE[bh * Tq + q0 + i] = (l > 0.f) ? static_cast<float>(sM[i] + log(static_cast<double>(l))) : -CUDART_INF_F;
  }
}

template <int BN>
size_t fwd_smem(int d, int dv) {
  return sizeof(double) * (BM * (BN + 1) + BM) +
         sizeof(float) * (BM * (d + 1) + BN * (d + 1) + BN * dv + BM * BN + 2 * BM);
}

template <int BN>
cudaError_t fwd_launch(const LaunchFwd& a) {
  const size_t smem = fwd_smem<BN>(a.p.d, a.p.dv);
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.p.Tq + BM - 1) / BM, a.p.B * a.p.H);
  fwd_kernel<BN><<<grid, NT, smem, a.stream>>>(static_cast<const float*>(a.Q), static_cast<const float*>(a.K),
                                               static_cast<const float*>(a.V), static_cast<float*>(a.O),
                                               a.LSE, a.p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward

constexpr int BNB = 32;   // keys per tile in the backward kernels

struct BwdArgs {
  const float* Q;
  const float* K;
  const float* V;
  const float* dO;
  const float* LSE;
  const float* D;
  float* dQ;
  float* dK;
  float* dV;
  Problem p;
};

// P and dS of one (query tile, key tile) pair into shared memory.
//   P_ij  = exp(s_ij - LSE_i)          (s_ij in fp64, blocked -> 0)
//   dS_ij = P_ij * (dO_i . V_j - D_i)
__device__ __forceinline__ void tile_p_ds(const float* sQ, const float* sK, const float* sV, const float* sdO,
                                          const float* sLse, const float* sD, float* sP, float* sdS, int q0,
                                          int kv0, const Problem& p) {
  const int d = p.d, dv = p.dv;
  for (int e = threadIdx.x; e < BM * BNB; e += NT) {
    const int i = e / BNB, j = e - i * BNB;
    const int qi = q0 + i, kj = kv0 + j;
    const bool blocked = (qi >= p.Tq) || (kj >= p.Tk) || (p.causal && kj > qi) || (sLse[i] == -CUDART_INF_F);
    float pij = 0.f, dsij = 0.f;
    if (!blocked) {
      const double s = dot2(sQ + i * (d + 1), sK + j * (d + 1), d);
      pij = expf(static_cast<float>(s * static_cast<double>(p.scale) - static_cast<double>(sLse[i])));
      float dp = 0.f;
      const float* gr = sdO + i * (dv + 1);
      const float* vr = sV + j * (dv + 1);
      for (int c = 0; c < dv; ++c) dp = fmaf(gr[c], vr[c], dp);
      dsij = pij * (dp - sD[i]);
    }
    sP[i * (BNB + 1) + j] = pij;
    sdS[i * (BNB + 1) + j] = dsij;
  }
}

__device__ __forceinline__ void load_qrow_stats(float* sLse, float* sD, const float* LSE, const float* D,
                                                size_t bh, int q0, int Tq) {
  if (threadIdx.x < BM) {
    const int qi = q0 + threadIdx.x;
    sLse[threadIdx.x] = qi < Tq ? LSE[bh * Tq + qi] : -CUDART_INF_F;
    sD[threadIdx.x] = qi < Tq ? D[bh * padded_rows(Tq) + qi] : 0.f;
  }
}

// One CTA per (key tile, head): loops over the query tiles that see the key
// tile, accumulates dK and dV in registers, and (unless `with_dq` is 0) adds
// this key tile's share scale * dS K into dQ with fp32 atomics.
__global__ void __launch_bounds__(NT) dkdv_kernel(const BwdArgs a, int with_dq) {
  extern __shared__ float smem_f[];
  const Problem& p = a.p;
  const int d = p.d, dv = p.dv, Tq = p.Tq, Tk = p.Tk;
  float* sK = smem_f;                         // [BNB][d+1]
  float* sV = sK + BNB * (d + 1);             // [BNB][dv+1]
  float* sQ = sV + BNB * (dv + 1);            // [BM][d+1]
  float* sdO = sQ + BM * (d + 1);             // [BM][dv+1]
  float* sP = sdO + BM * (dv + 1);            // [BM][BNB+1]
  float* sdS = sP + BM * (BNB + 1);           // [BM][BNB+1]
  float* sLse = sdS + BM * (BNB + 1);         // [BM]
  float* sD = sLse + BM;                      // [BM]

  const int kv0 = blockIdx.x * BNB;
  const size_t bh = blockIdx.y;
  for (int e = threadIdx.x; e < BNB * d; e += NT) {
    const int r = e / d, c = e - r * d;
    sK[r * (d + 1) + c] = (kv0 + r < Tk) ? a.K[(bh * Tk + kv0 + r) * d + c] : 0.f;
  }
  for (int e = threadIdx.x; e < BNB * dv; e += NT) {
    const int r = e / dv, c = e - r * dv;
    sV[r * (dv + 1) + c] = (kv0 + r < Tk) ? a.V[(bh * Tk + kv0 + r) * dv + c] : 0.f;
  }
  constexpr int PER = (BNB * MAXD + NT - 1) / NT;
  float accK[PER], accV[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) accK[k] = accV[k] = 0.f;

  const int qt0 = p.causal ? kv0 / BM : 0;
  const int n_qt = (Tq + BM - 1) / BM;
  for (int qt = qt0; qt < n_qt; ++qt) {
    const int q0 = qt * BM;
    __syncthreads();
    for (int e = threadIdx.x; e < BM * d; e += NT) {
      const int r = e / d, c = e - r * d;
      sQ[r * (d + 1) + c] = (q0 + r < Tq) ? a.Q[(bh * Tq + q0 + r) * d + c] : 0.f;
    }
    for (int e = threadIdx.x; e < BM * dv; e += NT) {
      const int r = e / dv, c = e - r * dv;
      sdO[r * (dv + 1) + c] = (q0 + r < Tq) ? a.dO[(bh * Tq + q0 + r) * dv + c] : 0.f;
    }
    load_qrow_stats(sLse, sD, a.LSE, a.D, bh, q0, Tq);
    __syncthreads();
    tile_p_ds(sQ, sK, sV, sdO, sLse, sD, sP, sdS, q0, kv0, p);
    __syncthreads();
    // dV_j += sum_i P_ij dO_i ; dK_j += sum_i dS_ij Q_i
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = threadIdx.x + k * NT;
      if (e < BNB * dv) {
        const int j = e / dv, c = e - j * dv;
        float s = accV[k];
        for (int i = 0; i < BM; ++i) s = fmaf(sP[i * (BNB + 1) + j], sdO[i * (dv + 1) + c], s);
        accV[k] = s;
      }
      if (e < BNB * d) {
        const int j = e / d, c = e - j * d;
        float s = accK[k];
        for (int i = 0; i < BM; ++i) s = fmaf(sdS[i * (BNB + 1) + j], sQ[i * (d + 1) + c], s);
        accK[k] = s;
      }
    }
    if (with_dq) {
      // dQ_i += scale * sum_j dS_ij K_j
      for (int e = threadIdx.x; e < BM * d; e += NT) {
        const int i = e / d, c = e - i * d;
        if (q0 + i >= Tq) continue;
        float s = 0.f;
        for (int j = 0; j < BNB; ++j) s = fmaf(sdS[i * (BNB + 1) + j], sK[j * (d + 1) + c], s);
        atomicAdd(a.dQ + (bh * Tq + q0 + i) * d + c, s * p.scale);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int e = threadIdx.x + k * NT;
    if (e < BNB * dv) {
      const int j = e / dv, c = e - j * dv;
      if (kv0 + j < Tk) a.dV[(bh * Tk + kv0 + j) * dv + c] = accV[k];
    }
    if (e < BNB * d) {
      const int j = e / d, c = e - j * d;
      if (kv0 + j < Tk) a.dK[(bh * Tk + kv0 + j) * d + c] = accK[k] * p.scale;
    }
  }
}

// Deterministic dQ: one CTA per (query tile, head) loops over key tiles in a
// fixed order and writes dQ once.
__global__ void __launch_bounds__(NT) dq_kernel(const BwdArgs a) {
  extern __shared__ float smem_f[];
  const Problem& p = a.p;
  const int d = p.d, dv = p.dv, Tq = p.Tq, Tk = p.Tk;
  float* sQ = smem_f;                         // [BM][d+1]
  float* sdO = sQ + BM * (d + 1);             // [BM][dv+1]
  float* sK = sdO + BM * (dv + 1);            // [BNB][d+1]
  float* sV = sK + BNB * (d + 1);             // [BNB][dv+1]
  float* sP = sV + BNB * (dv + 1);            // [BM][BNB+1]
  float* sdS = sP + BM * (BNB + 1);           // [BM][BNB+1]
  float* sLse = sdS + BM * (BNB + 1);
  float* sD = sLse + BM;

  const int q0 = blockIdx.x * BM;
  const size_t bh = blockIdx.y;
  for (int e = threadIdx.x; e < BM * d; e += NT) {
    const int r = e / d, c = e - r * d;
    sQ[r * (d + 1) + c] = (q0 + r < Tq) ? a.Q[(bh * Tq + q0 + r) * d + c] : 0.f;
  }
  for (int e = threadIdx.x; e < BM * dv; e += NT) {
    const int r = e / dv, c = e - r * dv;
    sdO[r * (dv + 1) + c] = (q0 + r < Tq) ? a.dO[(bh * Tq + q0 + r) * dv + c] : 0.f;
  }
  load_qrow_stats(sLse, sD, a.LSE, a.D, bh, q0, Tq);
  constexpr int PER = (BM * MAXD + NT - 1) / NT;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  int n_kt = (Tk + BNB - 1) / BNB;
  if (p.causal) n_kt = min(n_kt, (q0 + BM - 1) / BNB + 1);
  for (int kt = 0; kt < n_kt; ++kt) {
    const int kv0 = kt * BNB;
    __syncthreads();
    for (int e = threadIdx.x; e < BNB * d; e += NT) {
      const int r = e / d, c = e - r * d;
      sK[r * (d + 1) + c] = (kv0 + r < Tk) ? a.K[(bh * Tk + kv0 + r) * d + c] : 0.f;
    }
    for (int e = threadIdx.x; e < BNB * dv; e += NT) {
      const int r = e / dv, c = e - r * dv;
      sV[r * (dv + 1) + c] = (kv0 + r < Tk) ? a.V[(bh * Tk + kv0 + r) * dv + c] : 0.f;
    }
    __syncthreads();
    tile_p_ds(sQ, sK, sV, sdO, sLse, sD, sP, sdS, q0, kv0, p);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = threadIdx.x + k * NT;
      if (e < BM * d) {
        const int i = e / d, c = e - i * d;
        float s = acc[k];
        for (int j = 0; j < BNB; ++j) s = fmaf(sdS[i * (BNB + 1) + j], sK[j * (d + 1) + c], s);
        acc[k] = s;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int e = threadIdx.x + k * NT;
    if (e < BM * d) {
      const int i = e / d, c = e - i * d;
      if (q0 + i < Tq) a.dQ[(bh * Tq + q0 + i) * d + c] = acc[k] * p.scale;
    }
  }
}

size_t bwd_smem(int d, int dv) {
  return sizeof(float) * (BNB * (d + 1) + BNB * (dv + 1) + BM * (d + 1) + BM * (dv + 1) + 2 * BM * (BNB + 1) +
                          2 * BM);
}

}  // namespace simt

size_t fwd_f32_smem_bytes(int block_n, int d, int dv) {
  switch (block_n) {
    case 32: return simt::fwd_smem<32>(d, dv);
    case 128: return simt::fwd_smem<128>(d, dv);
    default: return simt::fwd_smem<64>(d, dv);
  }
}

cudaError_t launch_fwd_f32(const LaunchFwd& a) {
  switch (a.block_n) {
    case 32: return simt::fwd_launch<32>(a);
    case 128: return simt::fwd_launch<128>(a);
    default: return simt::fwd_launch<64>(a);
  }
}

cudaError_t launch_bwd_f32(const LaunchBwd& a) {
  const Problem& p = a.p;
  cudaError_t e = cudaSuccess;
  if (a.phase == 0 || a.phase == 1) {
    // D = rowsum(dO o O); dQ zeroed when it is accumulated with atomics.
    e = launch_bwd_preprocess(p, a.O, a.dO, a.LSE, 4, a.D, a.NLSE2,
                              a.deterministic ? nullptr : static_cast<float*>(a.dQ), p.d, a.num_sms, a.stream);
    if (e != cudaSuccess) return e;
  }
  const bool kv = a.phase == 0 || a.phase == 2 || a.phase == 4;
  const bool q = a.deterministic && (a.phase == 0 || a.phase == 2 || a.phase == 5);
  if (!kv && !q) return cudaSuccess;
  simt::BwdArgs b{static_cast<const float*>(a.Q), static_cast<const float*>(a.K), static_cast<const float*>(a.V),
                  static_cast<const float*>(a.dO), a.LSE, a.D, static_cast<float*>(a.dQ),
                  static_cast<float*>(a.dK), static_cast<float*>(a.dV), p};
  const size_t smem = simt::bwd_smem(p.d, p.dv);
  e = cudaFuncSetAttribute(simt::dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(simt::dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (kv && p.Tk > 0) {
    dim3 g1((p.Tk + simt::BNB - 1) / simt::BNB, p.B * p.H);
    simt::dkdv_kernel<<<g1, simt::NT, smem, a.stream>>>(b, a.deterministic ? 0 : 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (q) {
    dim3 g2((p.Tq + simt::BM - 1) / simt::BM, p.B * p.H);
    simt::dq_kernel<<<g2, simt::NT, smem, a.stream>>>(b);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace attn
