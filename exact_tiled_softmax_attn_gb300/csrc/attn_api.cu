// C-ABI layer: argument validation, tensor-map construction, workspace
// layout, dispatch to the kernels, and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "attn.h"
#include "common.cuh"
#include "launch.h"
#include "simt.h"
#include "ptx.cuh"

namespace attn {
namespace {

// Device status word shared by every kernel launched through this library.
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int num_sms = 0;
  int l2_bytes = 0;
  uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

thread_local int t_last_cuda_error = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

attn_status_t cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

// Per-device facts, resolved once per device with that device current.
attn_status_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  DeviceInfo& di = g_dev[dev];
  std::call_once(di.once, [&] {
    di.err = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (di.err == cudaSuccess) di.err = cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev);
    if (di.err == cudaSuccess) di.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.status), g_device_status);
  });
  if (di.err != cudaSuccess) return cuda_fail(di.err);
  *out = &di;
  return ATTN_OK;
}

attn_status_t encoder(EncodeTiledFn* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!g_encode) return ATTN_ERR_CUDA;
  *fn = g_encode;
  return ATTN_OK;
}

// 3-D map over a [planes, rows, inner] array with 128-byte swizzled boxes of
// box_rows rows x (128 bytes of elements): 64 bf16 or 32 fp32. Rows past
// `rows` read as zero within each plane (and are not written by reduces).
attn_status_t make_map(CUtensorMap* m, const void* base, int inner, int rows, int planes, bool f32 = false,
                       unsigned box_rows = 128) {
  EncodeTiledFn enc;
  attn_status_t s = encoder(&enc);
  if (s != ATTN_OK) return s;
  const cuuint64_t es = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(planes)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * es,
                                 static_cast<cuuint64_t>(inner) * es * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {f32 ? 32u : 64u, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

size_t elem_size(attn_dtype_t dt) { return dt == ATTN_BF16 ? 2 : 4; }

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range range(const void* p, size_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + bytes};
}

// bf16 shapes. The forward takes d and dv in [8, 256], multiples of 8 (a row
// of Q, K, V or O is then a whole number of 16-byte TMA and store units): the
// kernels run on the next tile width up (64, 128 or 256 columns), the tensor
// maps read the missing columns of Q, K and V as zeros, which leave S and the
// first dv columns of O unchanged, and the epilogues write dv columns. The
// backward kernels take d, dv in {64, 128}, or d = 256 with dv in {64, 128,
// 256}; other widths run on zero-padded copies (bf16_bwd_padded).
bool bf16_fwd_shape(int d, int dv) { return d % 8 == 0 && dv % 8 == 0 && d <= 256 && dv <= 256; }
bool bf16_bwd_shape(int d, int dv) {
  return ((d == 64 || d == 128) && (dv == 64 || dv == 128)) || (d == 256 && (dv == 64 || dv == 128 || dv == 256));
}
// the d = 256 backward (bwd_d256.cu): no fp32 dQ accumulator, no dQ splits
bool bf16_bwd_wide(int d) { return d > 128; }
// rows wider than 128 columns go to the d = 256 forward kernel
bool bf16_wide(int d, int dv) { return d > 128 || dv > 128; }

attn_status_t check_common(int B, int H, int Tq, int Tk, int d, int dv, float scale, int causal, attn_dtype_t dt) {
  if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || d <= 0 || dv <= 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (dt != ATTN_F32 && dt != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (dt == ATTN_F32) {
    if (d > 256 || dv > 256) return ATTN_ERR_UNSUPPORTED;
  } else if (!bf16_fwd_shape(d, dv)) {
    return ATTN_ERR_UNSUPPORTED;
  }
  // every index of every tensor must fit the kernels' 64-bit arithmetic and
  // the per-head row counts must fit int (TMA coordinates are int32)
  const double elems = static_cast<double>(B) * H * (Tq > Tk ? Tq : Tk) * (d > dv ? d : dv);
  if (elems > 9.0e15) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status_t check_ptr(const void* p, size_t bytes, size_t align) {
  if (bytes == 0) return ATTN_OK;  // empty tensors may be NULL
  if (p == nullptr) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(p) % align) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Key splits for `units` work units of nkb key tiles each, one CTA per unit
// and key range on `slots` SMs: the time of S splits is taken as the waves of
// units * S CTAs times the key tiles of a split, and the result is the
// smallest S within 5 % of the best, with at least two key tiles per split
// and at most 64 splits.
int wave_splits(long long units, int nkb, int slots) {
  if (units <= 0 || slots <= 0 || nkb < 4) return 1;
  const int smax = nkb / 2 < 64 ? nkb / 2 : 64;
  auto cost = [&](int s) {   // waves x key tiles per split
    const long long cs = (nkb + s - 1) / s, se = (nkb + cs - 1) / cs;
    return static_cast<double>((units * se + slots - 1) / slots) * static_cast<double>(cs);
  };
  double best = cost(1);
  for (int s = 2; s <= smax; ++s) best = cost(s) < best ? cost(s) : best;
  int S = 1;
  while (S < smax && cost(S) > 1.05 * best) ++S;
  return S;
}

struct BwdLayout {
  size_t lse2_off, d_off, acc_off, acc_bytes, sched_off, total;
  int dq_splits, dq_split_tiles;   // split deterministic dQ (bf16): acc holds the partials
};
// The deterministic bf16 dQ kernel runs one unit per 128-row query tile; when
// a problem has few query tiles against many key tiles (fewer units than
// half a GB300's 152 SMs, at least 8 key tiles), each query tile's keys are
// split into ranges so that at most 152 units run (one wave), each with at
// least 4 key tiles; at most 64 splits. A rule of the shapes only, so the workspace size
// needs no device.
// fp32: with at most 1 GiB of partials (f32_fused_dq) every 64-key tile is
// a range of its own, whose partial dQ the dK/dV kernel writes; otherwise
// the fp32 dQ kernel (one CTA per 64-row query tile) splits its units over
// ranges of 64-key tiles by the wave model of wave_splits on 152 SMs, also a
// rule of the shapes only.
constexpr int kDqSplitTargetUnits = 152;
void dq_split_count(int B, int H, int Tq, int Tk, int d, attn_dtype_t dt, int deterministic, int* S, int* cs) {
  if (dt == ATTN_F32) {
    const long long units = static_cast<long long>(B) * H * ((Tq + kF32SplitTile - 1) / kF32SplitTile);
    const int nkt = (Tk + kF32SplitTile - 1) / kF32SplitTile;
    if (deterministic && f32_fused_dq(B, H, Tq, Tk, d)) {
      *S = nkt;
      *cs = 1;
      return;
    }
    const int want = deterministic ? wave_splits(units, nkt, kDqSplitTargetUnits) : 1;
    *cs = want > 1 ? (nkt + want - 1) / want : nkt;
    *S = want > 1 ? (nkt + *cs - 1) / *cs : 1;
    return;
  }
  const long long units = static_cast<long long>(B) * H * ((Tq + 127) / 128);
  const int nkt = (Tk + 127) / 128;
  *S = 1;
  *cs = nkt;
  if (dt != ATTN_BF16 || !deterministic || units == 0 || units >= kDqSplitTargetUnits / 2 || nkt < 8) return;
  long long want = kDqSplitTargetUnits / units;   // one wave: units * S <= 152
  if (want > nkt / 4) want = nkt / 4;
  if (want > 64) want = 64;
  if (want < 2) return;
  *cs = (nkt + static_cast<int>(want) - 1) / static_cast<int>(want);
  *S = (nkt + *cs - 1) / *cs;
  if (*S < 2) {
    *S = 1;
    *cs = nkt;
  }
}

// Workspace: NLSE2 [B*H, Tq_pad] fp32 | D [B*H, Tq_pad] fp32 | (bf16 with fp32
// dQ accumulation) dQacc [B*H*Tq, d] fp32, or (bf16 deterministic with split
// dQ) the partials [S][B*H*Tq, d] fp32 | (bf16, d <= 128) 256 bytes for the
// two unit counters of the dQ and dK/dV kernels; each part 256-byte aligned.
BwdLayout bwd_layout(int B, int H, int Tq, int Tk, int d, attn_dtype_t dt, int deterministic) {
  BwdLayout L{};
  const size_t rows_pad = static_cast<size_t>(B) * H * padded_rows(Tq);
  const size_t part = round_up(rows_pad * sizeof(float), 256);
  dq_split_count(B, H, Tq, Tk, d, dt, deterministic, &L.dq_splits, &L.dq_split_tiles);
  L.lse2_off = 0;
  L.d_off = part;
  L.acc_off = 2 * part;
  const size_t acc = static_cast<size_t>(B) * H * Tq * d * sizeof(float);
  L.acc_bytes = (dt == ATTN_BF16 && !deterministic) ? acc : (L.dq_splits > 1 ? L.dq_splits * acc : 0);
  if (dt == ATTN_BF16 && bf16_bwd_wide(d)) {
    // the d = 256 kernels write dQ in one fixed-order pass whatever `deterministic` says
    L.acc_bytes = 0;
    L.dq_splits = 1;
    L.dq_split_tiles = (Tk + 127) / 128;
  }
  L.sched_off = round_up(L.acc_off + L.acc_bytes, 256);
  const size_t sched = (dt == ATTN_BF16 && !bf16_bwd_wide(d)) ? 256 : 0;
  L.total = rows_pad ? L.sched_off + sched : 0;
  return L;
}

// bf16 backward at other widths (multiples of 8 up to 256): Q, K, V, O and
// dO are copied into rows of the next width dp, dvp the kernels take, with
// zero columns, the backward runs on those copies, and the first d / dv
// columns of its gradients are copied out. The zero columns add nothing to
// S = QK^T, dP = dO V^T or D = rowsum(dO o O), so P and dS are those of the
// unpadded problem and the gradients' first columns are its gradients.
bool bf16_bwd_padded(int d, int dv) { return !bf16_bwd_shape(d, dv) && bf16_fwd_shape(d, dv); }

struct PadLayout {
  int dp, dvp;
  size_t q, k, v, o, dO, dq, dk, dv, inner, total;   // byte offsets in the workspace; inner: the backward's own
};
// Workspace of the padded backward: Qp | Kp | Vp | Op | dOp | dQp | dKp | dVp
// (bf16, rows of dp or dvp columns), each 256-byte aligned, then the
// workspace of the backward at (dp, dvp).
PadLayout pad_layout(int B, int H, int Tq, int Tk, int d, int dv, int deterministic) {
  PadLayout L{};
  // rows wider than 128 columns on either side run on the d = 256 kernels
  const bool wide = d > 128 || dv > 128;
  L.dp = wide ? 256 : (d <= 64 ? 64 : 128);
  L.dvp = dv <= 64 ? 64 : (dv <= 128 ? 128 : 256);
  const size_t bh = static_cast<size_t>(B) * H;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  L.q = take(bh * Tq * L.dp * 2);
  L.k = take(bh * Tk * L.dp * 2);
  L.v = take(bh * Tk * L.dvp * 2);
  L.o = take(bh * Tq * L.dvp * 2);
  L.dO = take(bh * Tq * L.dvp * 2);
  L.dq = take(bh * Tq * L.dp * 2);
  L.dk = take(bh * Tk * L.dp * 2);
  L.dv = take(bh * Tk * L.dvp * 2);
  L.inner = off;
  L.total = off + bwd_layout(B, H, Tq, Tk, L.dp, ATTN_BF16, deterministic).total;
  return L;
}

// Split-KV forward: effective number of key splits for a request, clamped to
// [1, min(key tiles, 64)]; the key tiles per split go to *split_tiles. A
// bf16 unit is a pair of 128-row query tiles for rows of up to 128 columns
// and one query tile for wider rows, with 128-key tiles; an fp32 unit is one
// 64-row query tile, with 64-key tiles (one CTA per SM either way). Request
// 0 picks the count: the time of S splits is taken as the waves of units * S
// CTAs over the SMs times the key tiles of a split, and S is the smallest
// count within 5 % of the best (at least two key tiles per split). A bf16
// problem with at least as many units as SMs does not split: its persistent
// forward spreads the units over the SMs itself.
int splitkv_count(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dt, int req, int num_sms,
                  int* split_tiles) {
  const bool f32 = dt == ATTN_F32;
  const int tile = f32 ? kF32SplitTile : 128;
  const int rows_per_unit = f32 ? kF32SplitTile : bf16_wide(d, dv) ? 128 : 256;
  const int nkb = (Tk + tile - 1) / tile;
  int S = req;
  if (nkb <= 1 || B == 0 || H == 0 || Tq == 0) {
    S = 1;
  } else if (req == 0) {
    const long long units = static_cast<long long>(B) * H * ((Tq + rows_per_unit - 1) / rows_per_unit);
    S = (!f32 && units >= num_sms) ? 1 : wave_splits(units, nkb, num_sms);
  }
  if (S > nkb) S = nkb;
  if (S > 64) S = 64;
  if (S < 1) S = 1;
  const int cs = (nkb + S - 1) / S;
  *split_tiles = cs;
  return nkb > 0 ? (nkb + cs - 1) / cs : 1;
}

struct SplitLayout {
  size_t lse_off, total;
};
// Workspace of the split-KV forward: Opart [S][B*H*Tq][dv] fp32 | LSEpart
// [S][B*H*Tq] (fp32 for bf16 problems, fp64 for fp32 ones), each part
// 256-byte aligned; nothing when S = 1.
SplitLayout split_layout(int B, int H, int Tq, int dv, int S, attn_dtype_t dt) {
  SplitLayout L{};
  if (S <= 1) return L;
  const size_t rows = static_cast<size_t>(B) * H * Tq;
  const size_t lse_bytes = dt == ATTN_F32 ? sizeof(double) : sizeof(float);
  L.lse_off = round_up(static_cast<size_t>(S) * rows * dv * sizeof(float), 256);
  L.total = L.lse_off + round_up(static_cast<size_t>(S) * rows * lse_bytes, 256);
  return L;
}

attn_status_t fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Tq,
                       int Tk, int d, int dv, float scale, int causal, attn_dtype_t dtype, int block_n,
                       int split_req, void* workspace, size_t workspace_bytes, void* stream) {
  attn_status_t s = check_common(B, H, Tq, Tk, d, dv, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  if (split_req < 0) return ATTN_ERR_INVALID_ARG;
  // the CUDA-core forward keeps a key tile of K and V rows in shared memory:
  // with d or dv above 128 a 128-key tile does not fit
  if (dtype == ATTN_F32 && fwd_f32_smem_bytes(block_n, d, dv) > 227 * 1024) return ATTN_ERR_UNSUPPORTED;
  const size_t es = elem_size(dtype);
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t align = dtype == ATTN_BF16 ? 16 : 4;
  const size_t bq = bh * Tq * d * es, bk = bh * Tk * d * es, bv = bh * Tk * dv * es, bo = bh * Tq * dv * es,
               bl = bh * Tq * 4;
  if ((s = check_ptr(Q, bq, align)) != ATTN_OK) return s;
  if ((s = check_ptr(K, bk, align)) != ATTN_OK) return s;
  if ((s = check_ptr(V, bv, align)) != ATTN_OK) return s;
  if ((s = check_ptr(O, bo, align)) != ATTN_OK) return s;
  if ((s = check_ptr(LSE, bl, 4)) != ATTN_OK) return s;
  const Range ro = range(O, bo), rl = range(LSE, bl);
  for (Range in : {range(Q, bq), range(K, bk), range(V, bv)})
    if (overlap(ro, in) || overlap(rl, in)) return ATTN_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return ATTN_ERR_INVALID_ARG;
  int split_tiles = 0, n_splits = 1;
  SplitLayout SL{};
  DeviceInfo* di = nullptr;
  if (split_req != 1) {
    // only the automatic choice needs the device (its SM count)
    if (split_req == 0 && (s = device_info(&di)) != ATTN_OK) return s;
    n_splits = splitkv_count(B, H, Tq, Tk, d, dv, dtype, split_req, di ? di->num_sms : 0, &split_tiles);
    SL = split_layout(B, H, Tq, dv, n_splits, dtype);
    if (SL.total > 0) {
      if (workspace == nullptr || workspace_bytes < SL.total || reinterpret_cast<uintptr_t>(workspace) % 256)
        return ATTN_ERR_WORKSPACE;
      const Range rw = range(workspace, SL.total);
      for (Range other : {range(Q, bq), range(K, bk), range(V, bv), ro, rl})
        if (overlap(rw, other)) return ATTN_ERR_WORKSPACE;
    }
  }
  if (bh == 0 || Tq == 0) return ATTN_OK;

  if (di == nullptr && (s = device_info(&di)) != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Problem p{B, H, Tq, Tk, d, dv, scale, causal};
  if (Tk == 0) {
    cudaError_t e = launch_fill_empty_fwd(p, O, LSE, static_cast<int>(es), st);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  LaunchFwd a{};
  a.p = p;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.LSE = LSE;
  a.status = di->status;
  a.num_sms = di->num_sms;
  a.block_n = block_n;
  a.n_splits = n_splits;
  a.split_tiles = split_tiles;
  if (n_splits > 1) {
    a.Opart = static_cast<float*>(workspace);
    // fp32 problems: fp64 log-sum-exps (the fp32 kernels cast the pointer back)
    a.LSEpart = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + SL.lse_off);
  }
  a.stream = st;
  cudaError_t e;
  if (dtype == ATTN_F32) {
    e = launch_fwd_f32(a);
    if (e == cudaSuccess && n_splits > 1)
      e = launch_splitkv_merge_f32(p, a.Opart, reinterpret_cast<const double*>(a.LSEpart), n_splits, split_tiles,
                                   kF32SplitTile, static_cast<float*>(O), LSE, di->num_sms, st);
  } else {
    // Rows wider than 128 columns: on CTA pairs (each CTA loads 64-key
    // halves of K and 128-key tiles of half of V's columns) unless the keys
    // are split or V is 64 columns wide; otherwise the one-CTA kernel, which
    // loads V by 64-key halves of its 128-key tiles.
    const bool wide = bf16_wide(d, dv);
    const bool pair = wide && n_splits == 1 && dv > 64;
    const unsigned k_rows = pair ? 64u : 128u;
    const unsigned v_rows = wide && !pair ? 64u : 128u;
    CUtensorMap mq, mk, mv;
    if ((s = make_map(&mq, Q, d, Tq, static_cast<int>(bh))) != ATTN_OK) return s;
    if ((s = make_map(&mk, K, d, Tk, static_cast<int>(bh), false, k_rows)) != ATTN_OK) return s;
    if ((s = make_map(&mv, V, dv, Tk, static_cast<int>(bh), false, v_rows)) != ATTN_OK) return s;
    a.tmQ = &mq;
    a.tmK = &mk;
    a.tmV = &mv;
    e = pair ? launch_fwd_bf16_d256_pair(a) : wide ? launch_fwd_bf16_d256(a) : launch_fwd_bf16(a);
    if (e == cudaSuccess && n_splits > 1)
      e = launch_splitkv_merge(p, a.Opart, a.LSEpart, n_splits, split_tiles, O, LSE, di->num_sms, st);
  }
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- self-test

__global__ void wait_timeout_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_word;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_word = 0u;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ptx::WaitCtx w{&abort_word, status, 15u};
    ptx::mbar_wait(&bar, 0u, w, limit_ns);  // nobody arrives: gives up after limit_ns
  }
  __syncthreads();
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

attn_status_t attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Tq,
                       int Tk, int d, int dv, float scale, int causal, attn_dtype_t dtype, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, Tq, Tk, d, dv, scale, causal, dtype, 64, 1, nullptr, 0, stream);
}

int attn_fwd_splitkv_splits(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype, int num_splits) {
  if (check_common(B, H, Tq, Tk, d, dv, 1.0f, 0, dtype) != ATTN_OK || num_splits < 0) return -1;
  int num_sms = 0;
  if (num_splits == 0) {
    DeviceInfo* di;
    if (device_info(&di) != ATTN_OK) return -1;
    num_sms = di->num_sms;
  }
  int cs;
  return splitkv_count(B, H, Tq, Tk, d, dv, dtype, num_splits, num_sms, &cs);
}

size_t attn_fwd_splitkv_workspace_size(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype,
                                       int num_splits) {
  const int S = attn_fwd_splitkv_splits(B, H, Tq, Tk, d, dv, dtype, num_splits);
  if (S < 1) return 0;
  return split_layout(B, H, Tq, dv, S, dtype).total;
}

attn_status_t attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                               int Tq, int Tk, int d, int dv, float scale, int causal, attn_dtype_t dtype,
                               int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, Tq, Tk, d, dv, scale, causal, dtype, 64, num_splits, workspace,
                  workspace_bytes, stream);
}

attn_status_t attn_fwd_f32_blocked(const float* Q, const float* K, const float* V, float* O, float* LSE, int B,
                                   int H, int Tq, int Tk, int d, int dv, float scale, int causal, int block_n,
                                   void* stream) {
  if (block_n != 32 && block_n != 64 && block_n != 128) return ATTN_ERR_UNSUPPORTED;
  return fwd_impl(Q, K, V, O, LSE, B, H, Tq, Tk, d, dv, scale, causal, ATTN_F32, block_n, 1, nullptr, 0, stream);
}

size_t attn_bwd_workspace_size(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype,
                               int deterministic) {
  if (check_common(B, H, Tq, Tk, d, dv, 1.0f, 0, dtype) != ATTN_OK) return 0;
  if (dtype == ATTN_BF16 && !bf16_bwd_shape(d, dv)) {
    if (!bf16_bwd_padded(d, dv) || (deterministic != 0 && deterministic != 1)) return 0;   // no bf16 backward there
    return pad_layout(B, H, Tq, Tk, d, dv, deterministic).total;
  }
  return bwd_layout(B, H, Tq, Tk, d, dtype, deterministic).total;
}

int attn_bwd_dq_splits(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype, int deterministic) {
  if (check_common(B, H, Tq, Tk, d, dv, 1.0f, 0, dtype) != ATTN_OK) return -1;
  if (dtype == ATTN_BF16 && !bf16_bwd_shape(d, dv) && !bf16_bwd_padded(d, dv)) return -1;
  if (deterministic != 0 && deterministic != 1) return -1;
  // the width the backward runs at (the padded one for other bf16 widths)
  const int d_run =
      dtype == ATTN_BF16 && bf16_bwd_padded(d, dv) ? pad_layout(B, H, Tq, Tk, d, dv, deterministic).dp : d;
  return bwd_layout(B, H, Tq, Tk, d_run, dtype, deterministic).dq_splits;
}

}  // extern "C"

namespace attn {
namespace {
attn_status_t bwd_impl(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                       void* dQ, void* dK, void* dV, int B, int H, int Tq, int Tk, int d, int dv, float scale,
                       int causal, attn_dtype_t dtype, int deterministic, void* workspace, size_t workspace_bytes,
                       int phase, void* stream) {
  attn_status_t s = check_common(B, H, Tq, Tk, d, dv, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  // the tensor-core backward kernels take d, dv in {64, 128} and d = 256 with
  // dv in {64, 128, 256}; other widths run on zero-padded copies (one call:
  // no phases)
  const bool padded = dtype == ATTN_BF16 && !bf16_bwd_shape(d, dv);
  if (padded && !bf16_bwd_padded(d, dv)) return ATTN_ERR_UNSUPPORTED;
  if (phase < 0 || phase > 6) return ATTN_ERR_INVALID_ARG;
  if (padded && phase != 0) return ATTN_ERR_UNSUPPORTED;
  // phase 6, the dQ pass on CTA pairs, exists for bf16 with d = 128 and deterministic dQ
  if (phase == 6 && (dtype != ATTN_BF16 || d != 128 || deterministic != 1)) return ATTN_ERR_UNSUPPORTED;
  if (deterministic != 0 && deterministic != 1) return ATTN_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t align = dtype == ATTN_BF16 ? 16 : 4;
  const size_t bq = bh * Tq * d * es, bk = bh * Tk * d * es, bv = bh * Tk * dv * es, bo = bh * Tq * dv * es,
               bl = bh * Tq * 4;
  const void* ins[6] = {Q, K, V, O, LSE, dO};
  const size_t in_bytes[6] = {bq, bk, bv, bo, bl, bo};
  for (int i = 0; i < 6; ++i)
    if ((s = check_ptr(ins[i], in_bytes[i], i == 4 ? 4 : align)) != ATTN_OK) return s;
  void* outs[3] = {dQ, dK, dV};
  const size_t out_bytes[3] = {bq, bk, bv};
  for (int i = 0; i < 3; ++i)
    if ((s = check_ptr(outs[i], out_bytes[i], align)) != ATTN_OK) return s;
  const BwdLayout L = bwd_layout(B, H, Tq, Tk, d, dtype, deterministic);
  const PadLayout PL = padded ? pad_layout(B, H, Tq, Tk, d, dv, deterministic) : PadLayout{};
  const size_t ws_total = padded ? PL.total : L.total;
  if (ws_total > 0) {
    if (workspace == nullptr || workspace_bytes < ws_total || reinterpret_cast<uintptr_t>(workspace) % 256)
      return ATTN_ERR_WORKSPACE;
  }
  // outputs must not overlap inputs, each other, or the workspace
  Range ro[4] = {range(dQ, bq), range(dK, bk), range(dV, bv), range(workspace, ws_total)};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlap(ro[i], range(ins[j], in_bytes[j]))) return i == 3 ? ATTN_ERR_WORKSPACE : ATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(ro[i], ro[j])) return ATTN_ERR_INVALID_ARG;
  }
  if (bh == 0) return ATTN_OK;

  DeviceInfo* di;
  if ((s = device_info(&di)) != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (Tq == 0 || Tk == 0) {
    // no (query, key) pair: every gradient is zero
    if (phase != 0 && phase != 2 && phase != 4) return ATTN_OK;
    if ((e = launch_zero(dQ, bq, st)) == cudaSuccess && (e = launch_zero(dK, bk, st)) == cudaSuccess)
      e = launch_zero(dV, bv, st);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  if (padded) {
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const long long rq = static_cast<long long>(bh) * Tq, rk = static_cast<long long>(bh) * Tk;
    const int ns = di->num_sms;
    if ((e = launch_pad_rows(Q, w + PL.q, rq, d, PL.dp, ns, st)) != cudaSuccess ||
        (e = launch_pad_rows(K, w + PL.k, rk, d, PL.dp, ns, st)) != cudaSuccess ||
        (e = launch_pad_rows(V, w + PL.v, rk, dv, PL.dvp, ns, st)) != cudaSuccess ||
        (e = launch_pad_rows(O, w + PL.o, rq, dv, PL.dvp, ns, st)) != cudaSuccess ||
        (e = launch_pad_rows(dO, w + PL.dO, rq, dv, PL.dvp, ns, st)) != cudaSuccess)
      return cuda_fail(e);
    s = bwd_impl(w + PL.q, w + PL.k, w + PL.v, w + PL.o, LSE, w + PL.dO, w + PL.dq, w + PL.dk, w + PL.dv, B, H, Tq,
                 Tk, PL.dp, PL.dvp, scale, causal, dtype, deterministic, w + PL.inner, PL.total - PL.inner, 0, stream);
    if (s != ATTN_OK) return s;
    if ((e = launch_crop_rows(w + PL.dq, dQ, rq, PL.dp, d, ns, st)) != cudaSuccess ||
        (e = launch_crop_rows(w + PL.dk, dK, rk, PL.dp, d, ns, st)) != cudaSuccess ||
        (e = launch_crop_rows(w + PL.dv, dV, rk, PL.dvp, dv, ns, st)) != cudaSuccess)
      return cuda_fail(e);
    return ATTN_OK;
  }
  LaunchBwd a{};
  a.p = Problem{B, H, Tq, Tk, d, dv, scale, causal};
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.LSE = LSE;
  a.dO = dO;
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.D = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.d_off);
  a.NLSE2 = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.lse2_off);
  float* acc = L.acc_bytes ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.acc_off) : nullptr;
  a.dQacc = deterministic ? nullptr : acc;
  a.dq_splits = L.dq_splits;
  a.dq_split_tiles = L.dq_split_tiles;
  a.dQpart = L.dq_splits > 1 ? acc : nullptr;
  a.deterministic = deterministic;
  a.sched = dtype == ATTN_BF16 && !bf16_bwd_wide(d)
                ? reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + L.sched_off)
                : nullptr;
  a.l2_bytes = static_cast<size_t>(di->l2_bytes);
  a.phase = phase;
  a.status = di->status;
  a.num_sms = di->num_sms;
  a.stream = st;
  if (dtype == ATTN_F32) {
    e = launch_bwd_f32(a);
  } else {
    CUtensorMap mq, mk, mv, mdo, mo, mdq;
    if ((s = make_map(&mq, Q, d, Tq, static_cast<int>(bh))) != ATTN_OK) return s;
    if ((s = make_map(&mk, K, d, Tk, static_cast<int>(bh))) != ATTN_OK) return s;
    if ((s = make_map(&mv, V, dv, Tk, static_cast<int>(bh))) != ATTN_OK) return s;
    if ((s = make_map(&mdo, dO, dv, Tq, static_cast<int>(bh))) != ATTN_OK) return s;
    if ((s = make_map(&mo, O, dv, Tq, static_cast<int>(bh))) != ATTN_OK) return s;
    a.tmQ = &mq;
    a.tmK = &mk;
    a.tmV = &mv;
    a.tmdO = &mdo;
    a.tmO = &mo;
    // the CTA-pair dQ kernel (phase 6) and the d = 256 kernels load 64-row halves of tiles
    CUtensorMap mq64, mk64, mv64, mdo64, mo64;
    if (phase == 6 || bf16_bwd_wide(d)) {
      if ((s = make_map(&mq64, Q, d, Tq, static_cast<int>(bh), false, 64)) != ATTN_OK) return s;
      if ((s = make_map(&mk64, K, d, Tk, static_cast<int>(bh), false, 64)) != ATTN_OK) return s;
      if ((s = make_map(&mv64, V, dv, Tk, static_cast<int>(bh), false, 64)) != ATTN_OK) return s;
      if ((s = make_map(&mdo64, dO, dv, Tq, static_cast<int>(bh), false, 64)) != ATTN_OK) return s;
      if ((s = make_map(&mo64, O, dv, Tq, static_cast<int>(bh), false, 64)) != ATTN_OK) return s;
      a.tmQ64 = &mq64;
      a.tmK64 = &mk64;
      a.tmV64 = &mv64;
      a.tmdO64 = &mdo64;
      a.tmO64 = &mo64;
    }
    a.tmdQacc = nullptr;
    if (a.dQacc) {
      if ((s = make_map(&mdq, a.dQacc, d, Tq, static_cast<int>(bh), true)) != ATTN_OK) return s;
      a.tmdQacc = &mdq;
    }
    e = bf16_bwd_wide(d) ? launch_bwd_bf16_d256(a) : launch_bwd_bf16(a);
  }
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
}  // namespace
}  // namespace attn

extern "C" {

attn_status_t attn_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                       const void* dO, void* dQ, void* dK, void* dV, int B, int H, int Tq, int Tk, int d, int dv,
                       float scale, int causal, attn_dtype_t dtype, int deterministic, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, Tq, Tk, d, dv, scale, causal, dtype, deterministic,
                  workspace, workspace_bytes, 0, stream);
}

attn_status_t attn_bwd_phase(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                             const void* dO, void* dQ, void* dK, void* dV, int B, int H, int Tq, int Tk, int d,
                             int dv, float scale, int causal, attn_dtype_t dtype, int deterministic, void* workspace,
                             size_t workspace_bytes, int phase, void* stream) {
  return bwd_impl(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, Tq, Tk, d, dv, scale, causal, dtype, deterministic,
                  workspace, workspace_bytes, phase, stream);
}

attn_status_t attn_device_status(void* stream) {
  DeviceInfo* di;
  attn_status_t s = device_info(&di);
  if (s != ATTN_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t v = 0;
  e = cudaMemcpy(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  const uint32_t zero = 0;
  e = cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v & ATTN_DEV_TIMEOUT) return ATTN_ERR_TIMEOUT;
  if (v) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_online_softmax_step(float* m, float* l, float* acc, const float* scores, const float* v_block,
                                       int n, int bs, int dv, void* stream) {
  if (n < 0 || bs < 0 || dv < 1 || dv > 512) return ATTN_ERR_INVALID_ARG;
  const size_t nn = static_cast<size_t>(n);
  const size_t bm = nn * 4, ba = nn * dv * 4, bsc = nn * bs * 4, bv = static_cast<size_t>(bs) * dv * 4;
  attn_status_t s;
  float* outs[3] = {m, l, acc};
  const size_t out_bytes[3] = {bm, bm, ba};
  for (int i = 0; i < 3; ++i)
    if ((s = check_ptr(outs[i], out_bytes[i], 4)) != ATTN_OK) return s;
  if ((s = check_ptr(scores, bsc, 4)) != ATTN_OK) return s;
  if ((s = check_ptr(v_block, bv, 4)) != ATTN_OK) return s;
  const Range ro[3] = {range(m, bm), range(l, bm), range(acc, ba)};
  for (int i = 0; i < 3; ++i) {
    if (overlap(ro[i], range(scores, bsc)) || overlap(ro[i], range(v_block, bv))) return ATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlap(ro[i], ro[j])) return ATTN_ERR_INVALID_ARG;
  }
  if (n == 0) return ATTN_OK;
  DeviceInfo* di;
  if ((s = device_info(&di)) != ATTN_OK) return s;
  const cudaError_t e =
      launch_online_softmax_step(m, l, acc, scores, v_block, n, bs, dv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

attn_status_t attn_selftest_wait_timeout(int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 5000) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di;
  attn_status_t s = device_info(&di);
  if (s != ATTN_OK) return s;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      di->status, static_cast<uint64_t>(limit_ms) * 1000000ull);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

const char* attn_strerror(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

int attn_last_cuda_error(void) { return t_last_cuda_error; }

int attn_version(void) { return (1 << 16) | 0; }

}  // extern "C"
