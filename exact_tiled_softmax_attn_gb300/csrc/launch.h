// Internal launch interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units. Not installed; the public header is include/attn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace attn {

struct LaunchFwd {
  Problem p;
  const CUtensorMap* tmQ;   // bf16 path only
  const CUtensorMap* tmK;
  const CUtensorMap* tmV;
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  float* LSE;
  uint32_t* status;
  int num_sms;
  int block_n;              // fp32 path: keys per tile (32, 64 or 128)
  // bf16 split-KV forward: n_splits > 1 key ranges of split_tiles 128-key
  // tiles each; partial outputs [n_splits][B*H*Tq][dv] and log-sum-exps
  // [n_splits][B*H*Tq] (fp32) instead of O and LSE
  int n_splits;
  int split_tiles;
  float* Opart;
  float* LSEpart;           // fp32 path: points at fp64 log-sum-exps (cast back to double*)
  cudaStream_t stream;
};

struct LaunchBwd {
  Problem p;
  const CUtensorMap* tmQ;   // bf16 path only
  const CUtensorMap* tmK;
  const CUtensorMap* tmV;
  const CUtensorMap* tmdO;
  const CUtensorMap* tmO;   // forward output O (bf16 deterministic dQ kernel: D of its rows)
  // 64-row boxes of Q, K, V, dO, O (bf16 deterministic dQ on CTA pairs, d = 128)
  const CUtensorMap* tmQ64;
  const CUtensorMap* tmK64;
  const CUtensorMap* tmV64;
  const CUtensorMap* tmdO64;
  const CUtensorMap* tmO64;
  const CUtensorMap* tmdQacc;  // fp32 dQ accumulator, 128 x 32 boxes (bf16 atomic path only)
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const float* LSE;
  const void* dO;
  void* dQ;
  void* dK;
  void* dV;
  float* D;                 // [B*H, Tq_pad] workspace, Tq_pad = Tq rounded up to 128
  float* NLSE2;             // [B*H, Tq_pad] workspace: -LSE * log2(e), -inf for padding / no-key rows
  float* dQacc;             // [B,H,Tq,d] fp32 workspace (bf16 atomic path), else null
  // bf16 deterministic path with few query tiles: the dQ kernel splits each
  // query tile's keys into dq_splits ranges of dq_split_tiles tiles, writes
  // fp32 partials to dQpart [dq_splits][B*H*Tq][d], and phase 3 adds them
  int dq_splits;
  int dq_split_tiles;
  float* dQpart;
  int deterministic;
  // bf16, d <= 128: two unit counters of the dQ and dK/dV kernels (zeroed
  // before each launch), and the device's L2 size, which sets how many heads'
  // tiles those kernels keep in flight at a time
  uint32_t* sched;
  size_t l2_bytes;
  int phase;                // 0 all; 1 preprocess; 2 main kernels (5 then 4); 3 dQ conversion / split reduction;
                            // 4 dK/dV kernel; 5 deterministic dQ kernel
  uint32_t* status;
  int num_sms;
  cudaStream_t stream;
};

// fp32 (SIMT; scores as float pairs from split rows or a compensated dot); d, dv <= 256
cudaError_t launch_fwd_f32(const LaunchFwd& a);
size_t fwd_f32_smem_bytes(int block_n, int d, int dv);   // dynamic shared memory of one forward CTA
cudaError_t launch_bwd_f32(const LaunchBwd& a);

// bf16 (tcgen05 / TMA)
cudaError_t launch_fwd_bf16(const LaunchFwd& a);
// d = 256 (dv 64, 128 or 256): one 128-row query tile per unit, 128-key
// tiles; tmK must be built with 128-row boxes and tmV with 64-row boxes
cudaError_t launch_fwd_bf16_d256(const LaunchFwd& a);
// The same on CTA pairs (two 128-row query tiles per cluster of two CTAs;
// dv above 64, no key split): tmQ with 128-row boxes, tmK with 64-row boxes,
// tmV with 128-row boxes
cudaError_t launch_fwd_bf16_d256_pair(const LaunchFwd& a);
cudaError_t launch_bwd_bf16(const LaunchBwd& a);
// d = 256 (dv 64, 128 or 256): a dQ kernel (which also forms D), then a dV
// and a dK kernel; needs the 64-row maps tmQ64, tmK64, tmV64, tmdO64, tmO64
// and the 128-row tmV, tmdO
cudaError_t launch_bwd_bf16_d256(const LaunchBwd& a);

// O, LSE from the split-KV partials (rows of query tile qt read the splits
// that hold at least one of its key tiles)
cudaError_t launch_splitkv_merge(const Problem& p, const float* Opart, const float* LSEpart, int n_splits,
                                 int split_tiles, void* O, float* LSE, int num_sms, cudaStream_t s);
// The same for the fp32 forward's key ranges (fp32 O, fp64 partial
// log-sum-exps; `tile` rows per query tile and keys per key tile of that
// forward)
cudaError_t launch_splitkv_merge_f32(const Problem& p, const float* Opart, const double* LSEpart, int n_splits,
                                     int split_tiles, int tile, float* O, float* LSE, int num_sms, cudaStream_t s);

// shared small kernels
cudaError_t launch_fill_empty_fwd(const Problem& p, void* O, float* LSE, int elem_bytes, cudaStream_t s);
cudaError_t launch_zero(void* ptr, size_t bytes, cudaStream_t s);
// bf16 rows of width w copied into rows of width wp >= w with zero columns
// (pad), or the first w columns of rows of width wp copied out (crop); w and
// wp multiples of 8, both buffers 16-byte aligned.
cudaError_t launch_pad_rows(const void* src, void* dst, long long rows, int w, int wp, int num_sms, cudaStream_t s);
cudaError_t launch_crop_rows(const void* src, void* dst, long long rows, int wp, int w, int num_sms, cudaStream_t s);
// One online-softmax step over n rows (fp32 state, fp64 arithmetic), dv <= 512.
cudaError_t launch_online_softmax_step(float* m, float* l, float* acc, const float* scores, const float* v, int n,
                                       int bs, int dv, cudaStream_t s);
// Rows of every head padded to a multiple of 128 (the backward's tile height).
__host__ __device__ inline int padded_rows(int T) { return (T + 127) / 128 * 128; }
// D = rowsum(dO o O) and NLSE2 = -LSE * log2(e) (-inf where LSE = -inf or the
// row is padding) in [B*H, Tq_pad] layout; optionally zeroes `zero_rows`
// ([B*H*Tq] rows of `zero_cols` floats).
cudaError_t launch_bwd_preprocess(const Problem& p, const void* O, const void* dO, const float* LSE, int elem_bytes,
                                  float* D, float* NLSE2, float* zero_rows, int zero_cols, int num_sms,
                                  cudaStream_t s);

}  // namespace attn
