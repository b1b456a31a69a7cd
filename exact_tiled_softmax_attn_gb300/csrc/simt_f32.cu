// fp32 attention forward and backward on the CUDA cores.
//
// Same tiled algorithm as the tensor-core path ("Tiled attention with an
// online softmax", section "Task"; gradients from "attention_backprop",
// sections "Gradient of V and P", "Gradient of S", "Gradient of Q and K"),
// for fp32 inputs of any head size up to 256.
//
// Precision: a score q.k is formed well beyond fp32 precision and kept as an
// unevaluated sum hi + lo of two floats; scale * (hi + lo) - m is formed from
// the exact product of hi and scale (one FMA gives its rounding error), so
// the argument of exp stays accurate even when the logits are in the
// thousands. Accumulating s in plain fp32 instead leaves a logit error of
// ~1e-5..1e-4 once |s| reaches the hundreds (keys scaled by +-40), which the
// softmax turns into output errors above 1e-5. Everything after the exponent
// (P, sums, P V, dP, dS, dQ, dK, dV) is fp32. Two ways of forming the score
// pair, chosen per kernel by whether its tiles fit in shared memory:
//  - split rows (rows up to 128 columns): every q and k row is split
//    exactly into a coarse part on a power-of-two grid set by the row's
//    largest entry plus a remainder; the coarse products then sum exactly in
//    fp32, and only the small cross terms round (3 FMAs per multiply-add);
//  - the compensated dot product Dot2 (10 FP32 instructions per
//    multiply-add) where the extra split rows do not fit (256 columns, and
//    128-key forward tiles of 128-column rows).
//
// Layout of the work: 256 threads per CTA as a 16 x 16 grid (ty, tx); a
// thread owns rows ty + 16 r (r < 4) of a 64-row tile and, in a score-shaped
// product, rows tx + 16 c of the tile it multiplies against (in a P V-shaped
// product, columns acc_col(tx, q) of the right-hand tile), so every product
// is a register tile of 4 x C results fed by 128-bit shared-memory loads,
// each carrying four steps of the reduction. Shared-memory rows are padded to
// W + 4 floats (W the tile width: 64, 128 or 256 columns, the smallest that
// holds d and dv): 16-byte aligned, and 8 consecutive rows start in 8
// different groups of four banks, so a warp's 128-bit loads of 16 rows take
// the two wavefronts their 256 bytes need. Columns from d (or dv) to W hold
// zeros. The products issue two-lane FMAs (fma.rn.f32x2) where their
// accumulators fit in registers. Each kernel runs one CTA per SM (its split
// tiles take most of the shared memory); a step's streamed tile loads into
// registers while the previous step's P V-shaped products run.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "simt.h"

namespace attn {
namespace simt {

constexpr int NT = 256;   // threads per CTA
constexpr int BM = 64;    // rows of the tile a CTA owns (queries; keys in the dK/dV kernel)

// Error-free transformations behind the compensated dot product of Ogita,
// Rump and Oishi ("Accurate Sum and Dot Product", SIAM J. Sci. Comput. 26(6),
// 2005, algorithm Dot2): a product splits exactly into p + e with one FMA,
// and the running sum is carried as s + c with Knuth's TwoSum, so the result
// is as accurate as a dot product accumulated in twice the fp32 precision,
// with fp32 instructions only (this GPU's fp64 rate is a small fraction of
// its fp32 rate). The _rn intrinsics keep the compiler from contracting the
// separate roundings the method relies on into FMAs.
__device__ __forceinline__ void dot2_step(float a, float b, float& s, float& c) {
  const float p = __fmul_rn(a, b);
  const float e = __fmaf_rn(a, b, -p);   // a b - p, exactly
  const float t = __fadd_rn(s, p);
  const float z = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(p, z));   // s + p - t, exactly
  s = t;
  c = __fadd_rn(c, __fadd_rn(err, e));
}

// scale * (hi + lo) as hi' + lo': hi' the rounded product, lo' its rounding
// error (exact, by FMA) plus scale * lo.
__device__ __forceinline__ void scale_pair(float hi, float lo, float scale, float& ph, float& pl) {
  ph = __fmul_rn(hi, scale);
  pl = __fadd_rn(__fmaf_rn(hi, scale, -ph), __fmul_rn(lo, scale));
}

// Exact split of a row x into x = hi + lo (the error-free splitting of
// Ozaki, Ogita, Oishi and Rump, "Error-free transformations of matrix
// multiplication by using fast routines of matrix multiplication and its
// applications", Numer. Algorithms 59, 2012, restated for rows of at most
// 256 entries). With E the exponent of the row's largest |x| (2^E <= max
// |x| < 2^(E+1)) and u = 2^(E-7), hi = rint(x / u) u is an integer multiple
// n u with |n| <= 256, and lo = x - hi, |lo| <= u / 2, is exact in fp32.
// For two split rows q, k of n <= 256 entries every partial sum of
// hq_i hk_i (over any subset of i) is an integer multiple of uq uk of at
// most 2^24 of them in magnitude, so the fp32 sum of the coarse products is
// exact in any order and grouping (as long as uq uk does not
// underflow, i.e. outside rows whose largest entries multiply to below
// ~2^-120); q.k = sum hq hk + sum (hq lk + lq k) with only the second sum,
// whose terms are 2^-8 of the scale of q.k, rounded.
// u and 1/u for a row whose largest |x| is m (>= 0): powers of two, both
// normal (rows below 2^-119 take u = 2^-126; inf and NaN are not split).
__device__ __forceinline__ void split_grid(float m, float& u, float& inv) {
  int eb = static_cast<int>((__float_as_uint(m) >> 23) & 0xffu);   // E + 127
  eb = min(max(eb, 8), 254);
  u = __uint_as_float(static_cast<uint32_t>(eb - 7) << 23);     // 2^(E - 7)
  inv = __uint_as_float(static_cast<uint32_t>(261 - eb) << 23);  // 2^(7 - E)
}

// ROWS rows of W columns on their way from global to shared memory, held in
// registers: warp w holds rows w, w + 8, ..., lane l columns l, l + 32, ...
// Loading and storing are separate steps, so that a tile's loads can be in
// flight while the CTA still computes on the previous tile.
template <int W, int ROWS>
struct RowRegs {
  static constexpr int NW = NT / 32, PER = W / 32, RW = ROWS / NW;
  static_assert(ROWS % NW == 0, "rows per warp");
  float v[RW][PER];

  // Rows [0, ROWS) of a [T][cols] fp32 block (src at its first row); rows at
  // or past `valid` and columns [cols, W) read as zeros.
  __device__ __forceinline__ void load(const float* src, int cols, int valid) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const int r = warp + NW * i;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int c = lane + 32 * j;
        v[i][j] = (r < valid && c < cols) ? src[static_cast<size_t>(r) * cols + c] : 0.f;
      }
    }
  }
  // To shared memory with rows of ld floats.
  __device__ __forceinline__ void store(float* dst, int ld) const {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int j = 0; j < PER; ++j) dst[(warp + NW * i) * ld + lane + 32 * j] = v[i][j];
  }
  // Each row split as above: hi to xh, lo to xl and, if xf is not null, x
  // itself to xf (shared memory, rows of ld floats).
  __device__ __forceinline__ void split(float* xf, float* xh, float* xl, int ld) const {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const int r = warp + NW * i;
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < PER; ++j) m = fmaxf(m, fabsf(v[i][j]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float u, inv;
      split_grid(m, u, inv);
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int c = lane + 32 * j;
        const float hi = __fmul_rn(rintf(__fmul_rn(v[i][j], inv)), u);
        xh[r * ld + c] = hi;
        xl[r * ld + c] = __fsub_rn(v[i][j], hi);
        if (xf != nullptr) xf[r * ld + c] = v[i][j];
      }
    }
  }
};

// Rows [0, ROWS) of a block loaded and split into shared memory at once.
template <int W, int ROWS>
__device__ __forceinline__ void load_split(float* xf, float* xh, float* xl, int ld, const float* src, int cols,
                                           int valid) {
  RowRegs<W, ROWS> x;
  x.load(src, cols, valid);
  x.split(xf, xh, xl, ld);
}

// Element i (0..3) of a float4; i is a constant once the loops are unrolled.
__device__ __forceinline__ float el(const float4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// The reduction products below read 4 consecutive reduction indices per
// 128-bit shared-memory load, over ceil(n / 4) * 4 indices: tiles are
// zero-filled to their width W (a multiple of 4), so the extra indices add 0.
// Each accumulator (each lane of a two-lane one) takes its terms in
// ascending index order, so every result is the same from run to run.

// a * b + c in each of two fp32 lanes, one instruction (sm_100 and later);
// each lane rounded as the scalar FMA
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
// elements (2h, 2h + 1) of a float4
__device__ __forceinline__ float2 pair(const float4& v, int h) { return h == 0 ? make_float2(v.x, v.y) : make_float2(v.z, v.w); }

// S[r][c] = sum_k A[ra + 16 r][k] B[cb + 16 c][k] over k < n from split
// rows, as s (the exact sum of the coarse products) + e (the cross terms):
// Ah, Al the A rows' parts, Bh, Bl the B rows'. FULL_A: e sums Al Bh + A Bl
// (A the unsplit A rows; B unused), else Ah Bl + Al B (A unused).
// Up to 4 columns per thread two-lane FMAs carry the even and the odd
// reduction indices in separate partial sums, added at the end (the coarse
// sums stay exact: any subset of the coarse products sums exactly); wider
// tiles (128-key forward tiles of 64-column rows) would not fit the doubled
// accumulators in registers and take one FMA per term.
template <int C, bool FULL_A>
__device__ __forceinline__ void split_tile(const float* A, const float* Ah, const float* Al, const float* B,
                                           const float* Bh, const float* Bl, int ld, int ra, int cb, int n,
                                           float (&s)[4][C], float (&e)[4][C]) {
  if constexpr (C > 4) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < C; ++c) s[r][c] = e[r][c] = 0.f;
    const int ao = ra * ld, bo = cb * ld, n4 = (n + 3) >> 2;
    for (int k = 0; k < 4 * n4; k += 4) {
      float4 ah[4], al[4], af[4], bh[C], bl[C], bf[C];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        ah[r] = ld4(Ah + ao + 16 * r * ld + k);
        al[r] = ld4(Al + ao + 16 * r * ld + k);
        if constexpr (FULL_A) af[r] = ld4(A + ao + 16 * r * ld + k);
      }
#pragma unroll
      for (int c = 0; c < C; ++c) {
        bh[c] = ld4(Bh + bo + 16 * c * ld + k);
        bl[c] = ld4(Bl + bo + 16 * c * ld + k);
        if constexpr (!FULL_A) bf[c] = ld4(B + bo + 16 * c * ld + k);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < C; ++c) {
            s[r][c] = __fmaf_rn(el(ah[r], i), el(bh[c], i), s[r][c]);   // exact
            if constexpr (FULL_A) {
              e[r][c] = __fmaf_rn(el(al[r], i), el(bh[c], i), e[r][c]);
              e[r][c] = __fmaf_rn(el(af[r], i), el(bl[c], i), e[r][c]);
            } else {
              e[r][c] = __fmaf_rn(el(ah[r], i), el(bl[c], i), e[r][c]);
              e[r][c] = __fmaf_rn(el(al[r], i), el(bf[c], i), e[r][c]);
            }
          }
    }
    return;
  }
  float2 s2[4][C], e2[4][C];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) s2[r][c] = e2[r][c] = make_float2(0.f, 0.f);
  const int ao = ra * ld, bo = cb * ld, n4 = (n + 3) >> 2;
#pragma unroll 2
  for (int k = 0; k < 4 * n4; k += 4) {
    float4 ah[4], al[4], af[4], bh[C], bl[C], bf[C];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ah[r] = ld4(Ah + ao + 16 * r * ld + k);
      al[r] = ld4(Al + ao + 16 * r * ld + k);
      if constexpr (FULL_A) af[r] = ld4(A + ao + 16 * r * ld + k);
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
      bh[c] = ld4(Bh + bo + 16 * c * ld + k);
      bl[c] = ld4(Bl + bo + 16 * c * ld + k);
      if constexpr (!FULL_A) bf[c] = ld4(B + bo + 16 * c * ld + k);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
          s2[r][c] = fma2(pair(ah[r], h), pair(bh[c], h), s2[r][c]);   // exact
          if constexpr (FULL_A) {
            e2[r][c] = fma2(pair(al[r], h), pair(bh[c], h), e2[r][c]);
            e2[r][c] = fma2(pair(af[r], h), pair(bl[c], h), e2[r][c]);
          } else {
            e2[r][c] = fma2(pair(ah[r], h), pair(bl[c], h), e2[r][c]);
            e2[r][c] = fma2(pair(al[r], h), pair(bf[c], h), e2[r][c]);
          }
        }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) {
      s[r][c] = __fadd_rn(s2[r][c].x, s2[r][c].y);
      e[r][c] = __fadd_rn(e2[r][c].x, e2[r][c].y);
    }
}

// split_tile<C, false> and dot_tile<C> of two row sets in one reduction
// loop (both products reduce over n): S from the split rows Ah, Al / B, Bh,
// Bl and X[r][c] = sum_k D[ra + 16 r][k] E[cb + 16 c][k]. Two-lane FMAs
// carry the even and the odd reduction indices in separate partial sums,
// added at the end (the coarse sums stay exact: any subset of the coarse
// products sums exactly).
template <int C>
__device__ __forceinline__ void split_dot_tile(const float* Ah, const float* Al, const float* B, const float* Bh,
                                               const float* Bl, const float* D, const float* E, int ld, int ra,
                                               int cb, int n, float (&s)[4][C], float (&e)[4][C],
                                               float (&x)[4][C]) {
  float2 s2[4][C], e2[4][C], x2[4][C];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) s2[r][c] = e2[r][c] = x2[r][c] = make_float2(0.f, 0.f);
  const int ao = ra * ld, bo = cb * ld, n4 = (n + 3) >> 2;
#pragma unroll 2
  for (int k = 0; k < 4 * n4; k += 4) {
    float4 ah[4], al[4], ad[4], bh[C], bl[C], bf[C], be[C];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ah[r] = ld4(Ah + ao + 16 * r * ld + k);
      al[r] = ld4(Al + ao + 16 * r * ld + k);
      ad[r] = ld4(D + ao + 16 * r * ld + k);
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
      bh[c] = ld4(Bh + bo + 16 * c * ld + k);
      bl[c] = ld4(Bl + bo + 16 * c * ld + k);
      bf[c] = ld4(B + bo + 16 * c * ld + k);
      be[c] = ld4(E + bo + 16 * c * ld + k);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
          s2[r][c] = fma2(pair(ah[r], h), pair(bh[c], h), s2[r][c]);   // exact
          e2[r][c] = fma2(pair(ah[r], h), pair(bl[c], h), e2[r][c]);
          e2[r][c] = fma2(pair(al[r], h), pair(bf[c], h), e2[r][c]);
          x2[r][c] = fma2(pair(ad[r], h), pair(be[c], h), x2[r][c]);
        }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) {
      s[r][c] = __fadd_rn(s2[r][c].x, s2[r][c].y);
      e[r][c] = __fadd_rn(e2[r][c].x, e2[r][c].y);
      x[r][c] = __fadd_rn(x2[r][c].x, x2[r][c].y);
    }
}

// S[r][c] = sum_k A[ra + 16 r][k] B[cb + 16 c][k] over k < n, by Dot2: hi in
// s, lo in e. A and B are shared-memory tiles with rows of `ld` floats.
template <int C>
__device__ __forceinline__ void dot2_tile(const float* A, const float* B, int ld, int ra, int cb, int n,
                                          float (&s)[4][C], float (&e)[4][C]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) s[r][c] = e[r][c] = 0.f;
  const float* a0 = A + ra * ld;
  const float* b0 = B + cb * ld;
  const int n4 = (n + 3) >> 2;
  for (int k = 0; k < 4 * n4; k += 4) {
    float4 a[4], b[C];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = ld4(a0 + 16 * r * ld + k);
#pragma unroll
    for (int c = 0; c < C; ++c) b[c] = ld4(b0 + 16 * c * ld + k);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) dot2_step(el(a[r], i), el(b[c], i), s[r][c], e[r][c]);
  }
}

// X[r][c] = sum_k A[ra + 16 r][k] B[cb + 16 c][k] over k < n (plain fp32).
template <int C>
__device__ __forceinline__ void dot_tile(const float* A, const float* B, int ld, int ra, int cb, int n,
                                         float (&x)[4][C]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) x[r][c] = 0.f;
  const float* a0 = A + ra * ld;
  const float* b0 = B + cb * ld;
  const int n4 = (n + 3) >> 2;
#pragma unroll 2
  for (int k = 0; k < 4 * n4; k += 4) {
    float4 a[4], b[C];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = ld4(a0 + 16 * r * ld + k);
#pragma unroll
    for (int c = 0; c < C; ++c) b[c] = ld4(b0 + 16 * c * ld + k);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) x[r][c] = fmaf(el(a[r], i), el(b[c], i), x[r][c]);
  }
}

// Column of the tile width held by a thread's q-th accumulator in the
// products below: four adjacent columns in every 64, so that a row of the
// right-hand tile is read with one 128-bit load per 64 columns.
__device__ __forceinline__ int acc_col(int tx, int q) { return 64 * (q >> 2) + 4 * tx + (q & 3); }

// acc[r][q] += sum_k P[ra + 16 r][k] V[k][acc_col(tx, q)] over k < n: P
// with rows of `ldp` floats, V with rows of `ldv` floats. Two adjacent
// columns share one two-lane FMA, P's element broadcast to both lanes.
template <int R, int Q>
__device__ __forceinline__ void acc_tile(const float* P, int ldp, const float* V, int ldv, int ra, int tx, int n,
                                         float (&acc)[R][Q]) {
  static_assert(Q % 4 == 0, "four columns per load");
  const float* p0 = P + ra * ldp;
  const float* v0 = V + 4 * tx;
  const int n4 = (n + 3) >> 2;
#pragma unroll 2
  for (int k = 0; k < 4 * n4; k += 4) {
    float4 a[R];
#pragma unroll
    for (int r = 0; r < R; ++r) a[r] = ld4(p0 + 16 * r * ldp + k);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 b[Q / 4];
#pragma unroll
      for (int g = 0; g < Q / 4; ++g) b[g] = ld4(v0 + (k + i) * ldv + 64 * g);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float2 ar = make_float2(el(a[r], i), el(a[r], i));
#pragma unroll
        for (int g = 0; g < Q / 4; ++g)
#pragma unroll
          for (int h = 0; h < 2; ++h) {   // columns 4g + 2h, 4g + 2h + 1: two lanes of one FMA
            const float2 t = fma2(ar, pair(b[g], h), make_float2(acc[r][4 * g + 2 * h], acc[r][4 * g + 2 * h + 1]));
            acc[r][4 * g + 2 * h] = t.x;
            acc[r][4 * g + 2 * h + 1] = t.y;
          }
      }
    }
  }
}

// Rows [r0, r0 + rows) of a [T][cols] fp32 matrix into shared memory with
// rows of ld floats: rows at or past `valid` and columns [cols, W) as zeros.
template <int W>
__device__ __forceinline__ void load_tile(float* dst, int ld, const float* src, int rows, int cols, int valid) {
  for (int e = threadIdx.x; e < rows * W; e += NT) {
    const int r = e / W, c = e - r * W;
    dst[r * ld + c] = (r < valid && c < cols) ? src[static_cast<size_t>(r) * cols + c] : 0.f;
  }
}

__device__ __forceinline__ float row_max16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float row_sum16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The tile width for head sizes d, dv: 64, 128 or 256 columns.
__host__ __device__ inline int tile_width(int d, int dv) {
  const int m = d > dv ? d : dv;
  return m <= 64 ? 64 : m <= 128 ? 128 : 256;
}

// ---------------------------------------------------------------- forward

// Key ranges of the split-KV forward: range z of a query tile holds its key
// tiles [z * tiles, (z + 1) * tiles); with n > 1 each (query tile, range)
// writes its own normalized O_z = A_z / l_z and LSE_z to Opart [n][B*H*Tq][dv]
// and LSEpart [n][B*H*Tq] (rows with no allowed key in the range: 0 and
// -inf), for the merge kernel. LSE_z stays in fp64: at logits in the
// thousands an fp32 LSE_z is off by up to 1e-4, and the merge weights
// exp(LSE_z - max) would carry that into O.
struct KeyRanges {
  int n, tiles;
  float* Opart;
  double* LSEpart;
};

// One CTA per (64-row query tile, head, key range); key tiles of BN keys in
// ascending order through the online softmax; O (4 x W/16 per thread) in
// registers. SPLIT: scores from split rows (Q whole and split, K split),
// else by Dot2.
template <int W, int BN, bool SPLIT>
__global__ void __launch_bounds__(NT, 1) fwd_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                 const float* __restrict__ V, float* __restrict__ O,
                                                 float* __restrict__ LSE, const Problem p, const KeyRanges ranges) {
  constexpr int LD = W + 4, LDP = BN + 4, NC = BN / 16, NQ = W / 16;
  extern __shared__ __align__(16) float smem_f[];
  float* sQ = smem_f;                              // [BM][LD]
  float* sQh = sQ + BM * LD;                       // split: [BM][LD] coarse parts of Q, then remainders
  float* sQl = sQh + BM * LD;
  float* sK = sQ + (SPLIT ? 3 : 1) * BM * LD;      // [BN][LD] K (split: its coarse parts, then remainders)
  float* sKl = sK + BN * LD;
  float* sV = sK + (SPLIT ? 2 : 1) * BN * LD;      // [BN][LD]
  float* sP = sV + BN * LD;                        // [BM][LDP]
  const int d = p.d, dv = p.dv, Tq = p.Tq, Tk = p.Tk;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int q0 = blockIdx.x * BM;
  const size_t bh = blockIdx.y;
  const float scale = p.scale;
  int n_kv = (Tk + BN - 1) / BN;
  if (p.causal) n_kv = min(n_kv, (q0 + BM - 1) / BN + 1);
  // this CTA's key tiles [j0, j1): a range past the causal limit has none
  // (the merge does not read it)
  const int j0 = blockIdx.z * ranges.tiles, j1 = ranges.n > 1 ? min(n_kv, j0 + ranges.tiles) : n_kv;
  if (j0 >= j1 && ranges.n > 1) return;

  if constexpr (SPLIT)
    load_split<W, BM>(sQ, sQh, sQl, LD, Q + (bh * Tq + q0) * d, d, Tq - q0);
  else
    load_tile<W>(sQ, LD, Q + (bh * Tq + q0) * d, BM, d, Tq - q0);
  float acc[4][NQ], m[4], l[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -CUDART_INF_F;
    l[r] = 0.f;
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[r][q] = 0.f;
  }

  // split rows: a key tile's K and V rows load into registers while the
  // previous tile's P V product runs
  RowRegs<W, BN> kr, vr;
  if constexpr (SPLIT) {
    kr.load(K + (bh * Tk + j0 * BN) * d, d, Tk - j0 * BN);
    vr.load(V + (bh * Tk + j0 * BN) * dv, dv, Tk - j0 * BN);
  }
  for (int jt = j0; jt < j1; ++jt) {
    const int kv0 = jt * BN;
    __syncthreads();   // the previous tile's P V is done with sK, sV, sP
    if constexpr (SPLIT) {
      kr.split(nullptr, sK, sKl, LD);
      vr.store(sV, LD);
    } else {
      load_tile<W>(sK, LD, K + (bh * Tk + kv0) * d, BN, d, Tk - kv0);
      load_tile<W>(sV, LD, V + (bh * Tk + kv0) * dv, BN, dv, Tk - kv0);
    }
    __syncthreads();
    float sh[4][NC], sl[4][NC];
    if constexpr (SPLIT)
      split_tile<NC, true>(sQ, sQh, sQl, nullptr, sK, sKl, LD, ty, tx, d, sh, sl);
    else
      dot2_tile<NC>(sQ, sK, LD, ty, tx, d, sh, sl);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int qi = q0 + ty + 16 * r;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int kj = kv0 + tx + 16 * c;
        float ph, pl;
        scale_pair(sh[r][c], sl[r][c], scale, ph, pl);
        const bool blocked = kj >= Tk || (p.causal && kj > qi);
        sh[r][c] = blocked ? -CUDART_INF_F : ph;
        sl[r][c] = blocked ? 0.f : pl;
        mx = fmaxf(mx, sh[r][c]);
      }
      mx = row_max16(mx);
      const float m_new = fmaxf(m[r], mx);
      const float ref = (m_new == -CUDART_INF_F) ? 0.f : m_new;   // the -inf rule
      const float corr = expf(m[r] - ref);                         // 0 when m = -inf
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const float pj = expf(__fadd_rn(__fsub_rn(sh[r][c], ref), sl[r][c]));
        sP[(ty + 16 * r) * LDP + tx + 16 * c] = pj;
        sum += pj;
      }
      l[r] = fmaf(l[r], corr, row_sum16(sum));
      m[r] = m_new;
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[r][q] *= corr;
    }
    __syncthreads();
    if constexpr (SPLIT) {
      if (jt + 1 < j1) {
        kr.load(K + (bh * Tk + kv0 + BN) * d, d, Tk - kv0 - BN);
        vr.load(V + (bh * Tk + kv0 + BN) * dv, dv, Tk - kv0 - BN);
      }
    }
    // acc += P V over the tile's keys (padding keys have P = 0 and V = 0)
    acc_tile<4, NQ>(sP, LDP, sV, LD, ty, tx, min(BN, Tk - kv0), acc);
  }
  // with key ranges, this range's partial state goes to the workspace
  const size_t rows = static_cast<size_t>(p.B) * p.H * Tq;
  float* Oout = ranges.n > 1 ? ranges.Opart + blockIdx.z * rows * dv : O;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int qi = q0 + ty + 16 * r;
    if (qi >= Tq) continue;
    const float inv = l[r] > 0.f ? 1.0f / l[r] : 0.f;
    float* orow = Oout + (bh * Tq + qi) * dv;
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (acc_col(tx, q) < dv) orow[acc_col(tx, q)] = acc[r][q] * inv;
    if (tx == 0) {
      const float ref = m[r] == -CUDART_INF_F ? 0.f : m[r];
      const double lse = l[r] > 0.f ? static_cast<double>(ref) + log(static_cast<double>(l[r])) : -CUDART_INF;
      if (ranges.n > 1)
        ranges.LSEpart[blockIdx.z * rows + bh * Tq + qi] = lse;
      else
        LSE[bh * Tq + qi] = static_cast<float>(lse);
    }
  }
}

constexpr size_t kSmemMax = 227 * 1024;

template <int W, int BN, bool SPLIT>
constexpr size_t fwd_smem_of() {
  return sizeof(float) * ((SPLIT ? 3 : 1) * BM * (W + 4) + (SPLIT ? 3 : 2) * BN * (W + 4) + BM * (BN + 4));
}
// split rows wherever their tiles fit
template <int W, int BN>
constexpr bool fwd_split() { return fwd_smem_of<W, BN, true>() <= kSmemMax; }
template <int W, int BN>
constexpr size_t fwd_smem() { return fwd_smem_of<W, BN, fwd_split<W, BN>()>(); }

template <int W, int BN>
cudaError_t fwd_launch(const LaunchFwd& a) {
  constexpr bool SP = fwd_split<W, BN>();
  constexpr size_t smem = fwd_smem<W, BN>();
  static_assert(smem <= kSmemMax, "shared memory");
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<W, BN, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int n_ranges = a.n_splits > 1 ? a.n_splits : 1;
  dim3 grid((a.p.Tq + BM - 1) / BM, a.p.B * a.p.H, n_ranges);
  // (fp32 problems: the split log-sum-exps are fp64, LSEpart points at them)
  const KeyRanges kr{n_ranges, a.split_tiles, a.Opart, reinterpret_cast<double*>(a.LSEpart)};
  fwd_kernel<W, BN, SP><<<grid, NT, smem, a.stream>>>(static_cast<const float*>(a.Q), static_cast<const float*>(a.K),
                                                  static_cast<const float*>(a.V), static_cast<float*>(a.O), a.LSE,
                                                  a.p, kr);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward

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
  // deterministic dQ over key ranges: count, 64-key tiles per range, partials
  int dq_splits;
  int dq_split_tiles;
  float* dQpart;
};

// P and dS of one score tile, for rows a + 16 r and columns b + 16 c of the
// tile (a thread's register tile): qi, kj the global query and key of each
// entry, lse and dd the query's LSE and D.
//   P = exp(scale s - LSE)   (0 where blocked)
//   dS = P (dP - D)
__device__ __forceinline__ void p_ds(float sh, float sl, float dp, float scale, float lse, float dd, bool blocked,
                                     float& pij, float& dsij) {
  float ph, pl;
  scale_pair(sh, sl, scale, ph, pl);
  pij = blocked ? 0.f : expf(__fadd_rn(__fsub_rn(ph, lse), pl));
  dsij = pij * (dp - dd);
}

// Four fp32 atomic adds to consecutive addresses in one instruction (sm_90+;
// the address 16-byte aligned).
__device__ __forceinline__ void red_add4(float* g, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(g), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// One CTA per (64-key tile, head): loops over the query tiles (BQ rows each)
// that see the key tile, computes S^T = K Q^T and dP^T = V dO^T for
// the tile, and accumulates dV += P^T dO and dK += dS^T Q in registers
// (rows of keys ty + 16 r). With `with_dq` it also forms this key tile's
// share scale * dS K of dQ: 1 adds it into dQ with fp32 atomics, 2 stores it
// into the key tile's own partial array a.dQpart[key tile] (dQ itself when
// there is one key tile), whose sum in key-tile order is dQ. SPLIT: scores
// from split rows (K split, Q whole and split), else by Dot2; with `with_dq`
// the split rows' K is also summed back into a whole copy for the dQ product.
template <int W, int BQ, bool SPLIT>
__global__ void __launch_bounds__(NT, 1) dkdv_kernel(const BwdArgs a, int with_dq) {
  constexpr int LD = W + 4, LDP = BQ + 4, NC = BQ / 16, NQ = W / 16;
  extern __shared__ __align__(16) float smem_f[];
  float* sK = smem_f;                            // [BM][LD] K (split: its coarse parts, then remainders)
  float* sKl = sK + BM * LD;
  float* sV = sK + (SPLIT ? 2 : 1) * BM * LD;    // [BM][LD]
  float* sQ = sV + BM * LD;                      // [BQ][LD] (split: then Q's coarse parts and remainders)
  float* sQh = sQ + BQ * LD;
  float* sQl = sQh + BQ * LD;
  float* sdO = sQ + (SPLIT ? 3 : 1) * BQ * LD;   // [BQ][LD]
  float* sPt = sdO + BQ * LD;     // [BM][LDP]  P^T: key rows, query columns
  float* sdSt = sPt + BM * LDP;                  // [BM][LDP]
  float* sLse = sdSt + BM * LDP;  // [BQ]
  float* sD = sLse + BQ;          // [BQ]
  float* sKf = sD + BQ;           // [BM][LD] split rows: K whole (coarse part + remainder), for the dQ product
  float* sdS = sKf + (SPLIT ? BM * LD : 0);   // [BQ][BM + 4] dS with query rows, for the dQ product
  const Problem& p = a.p;
  const int d = p.d, dv = p.dv, Tq = p.Tq, Tk = p.Tk;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int kv0 = blockIdx.x * BM;
  const size_t bh = blockIdx.y;
  const float scale = p.scale;

  if constexpr (SPLIT) {
    load_split<W, BM>(nullptr, sK, sKl, LD, a.K + (bh * Tk + kv0) * d, d, Tk - kv0);
    if (with_dq) {
      __syncthreads();
      for (int e = threadIdx.x; e < BM * LD; e += NT) sKf[e] = __fadd_rn(sK[e], sKl[e]);   // exact
    }
  }
  else
    load_tile<W>(sK, LD, a.K + (bh * Tk + kv0) * d, BM, d, Tk - kv0);
  load_tile<W>(sV, LD, a.V + (bh * Tk + kv0) * dv, BM, dv, Tk - kv0);
  float accV[4][NQ], accK[4][NQ];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < NQ; ++q) accV[r][q] = accK[r][q] = 0.f;

  const int qt0 = p.causal ? kv0 / BQ : 0;
  const int n_qt = (Tq + BQ - 1) / BQ;
  // split rows: a query step's Q and dO rows (and its LSE and D) load into
  // registers while the previous step's dV and dK products run
  RowRegs<W, BQ> qr, dor;
  float lse_n = -CUDART_INF_F, d_n = 0.f;
  auto load_step = [&](int q0) {
    qr.load(a.Q + (bh * Tq + q0) * d, d, Tq - q0);
    dor.load(a.dO + (bh * Tq + q0) * dv, dv, Tq - q0);
    if (threadIdx.x < BQ) {
      const int qi = q0 + threadIdx.x;
      lse_n = qi < Tq ? a.LSE[bh * Tq + qi] : -CUDART_INF_F;
      d_n = qi < Tq ? a.D[bh * padded_rows(Tq) + qi] : 0.f;
    }
  };
  if constexpr (SPLIT) load_step(qt0 * BQ);
  for (int qt = qt0; qt < n_qt; ++qt) {
    const int q0 = qt * BQ;
    __syncthreads();   // the previous step is done with sQ, sdO, sPt, sdSt
    if constexpr (SPLIT) {
      qr.split(sQ, sQh, sQl, LD);
      dor.store(sdO, LD);
      if (threadIdx.x < BQ) {
        sLse[threadIdx.x] = lse_n;
        sD[threadIdx.x] = d_n;
      }
    } else {
      load_tile<W>(sQ, LD, a.Q + (bh * Tq + q0) * d, BQ, d, Tq - q0);
      load_tile<W>(sdO, LD, a.dO + (bh * Tq + q0) * dv, BQ, dv, Tq - q0);
      if (threadIdx.x < BQ) {
        const int qi = q0 + threadIdx.x;
        sLse[threadIdx.x] = qi < Tq ? a.LSE[bh * Tq + qi] : -CUDART_INF_F;
        sD[threadIdx.x] = qi < Tq ? a.D[bh * padded_rows(Tq) + qi] : 0.f;
      }
    }
    __syncthreads();
    {
      float sh[4][NC], sl[4][NC], dp[4][NC];
      if constexpr (SPLIT) {
        // one loop for both products where it measured faster (128-column
        // rows; 64-column rows, which fit 64-query steps, were slower so)
        if (W >= 128 && d == dv) {
          split_dot_tile<NC>(sK, sKl, sQ, sQh, sQl, sV, sdO, LD, ty, tx, d, sh, sl, dp);
        } else {
          split_tile<NC, false>(nullptr, sK, sKl, sQ, sQh, sQl, LD, ty, tx, d, sh, sl);
          dot_tile<NC>(sV, sdO, LD, ty, tx, dv, dp);
        }
      } else {
        dot2_tile<NC>(sK, sQ, LD, ty, tx, d, sh, sl);
        dot_tile<NC>(sV, sdO, LD, ty, tx, dv, dp);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int kj = kv0 + ty + 16 * r;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int i = tx + 16 * c, qi = q0 + i;
          const float lse = sLse[i];
          const bool blocked = qi >= Tq || kj >= Tk || (p.causal && kj > qi) || lse == -CUDART_INF_F;
          float pij, dsij;
          p_ds(sh[r][c], sl[r][c], dp[r][c], scale, lse, sD[i], blocked, pij, dsij);
          sPt[(ty + 16 * r) * LDP + i] = pij;
          sdSt[(ty + 16 * r) * LDP + i] = dsij;
          if (with_dq) sdS[i * (BM + 4) + ty + 16 * r] = dsij;
        }
      }
    }
    __syncthreads();
    if constexpr (SPLIT) {
      if (qt + 1 < n_qt) load_step(q0 + BQ);
    }
    // dV_j += sum_i P_ij dO_i ; dK_j += sum_i dS_ij Q_i
    const int nq = min(BQ, Tq - q0);
    acc_tile<4, NQ>(sPt, LDP, sdO, LD, ty, tx, nq, accV);
    acc_tile<4, NQ>(sdSt, LDP, sQ, LD, ty, tx, nq, accK);
    if (with_dq) {
      // dQ_i += scale * sum_j dS_ij K_j, rows of queries ty + 16 r: a P V-shaped
      // product of the query-major dS tile and the whole K tile
      constexpr int RQ = BQ / 16;
      const float* kf = SPLIT ? sKf : sK;
      float t[RQ][NQ];
#pragma unroll
      for (int r = 0; r < RQ; ++r)
#pragma unroll
        for (int q = 0; q < NQ; ++q) t[r][q] = 0.f;
      acc_tile<RQ, NQ>(sdS, BM + 4, kf, LD, ty, tx, min(BM, Tk - kv0), t);
      float* dst = with_dq == 1 || a.dq_splits <= 1
                       ? a.dQ
                       : a.dQpart + static_cast<size_t>(blockIdx.x) * p.B * p.H * Tq * d;
      const bool vec = (d & 3) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
#pragma unroll
      for (int r = 0; r < RQ; ++r) {
        const int qi = q0 + ty + 16 * r;
        if (qi >= Tq) continue;
        float* row = dst + (bh * Tq + qi) * d;
#pragma unroll
        for (int g = 0; g < NQ / 4; ++g) {
          const int c = 64 * g + 4 * tx;
          const float4 v = make_float4(t[r][4 * g] * scale, t[r][4 * g + 1] * scale, t[r][4 * g + 2] * scale,
                                       t[r][4 * g + 3] * scale);
          if (vec && c + 3 < d) {
            if (with_dq == 1)
              red_add4(row + c, v.x, v.y, v.z, v.w);
            else
              *reinterpret_cast<float4*>(row + c) = v;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (c + e < d) {
                if (with_dq == 1)
                  atomicAdd(row + c + e, el(v, e));
                else
                  row[c + e] = el(v, e);
              }
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int kj = kv0 + ty + 16 * r;
    if (kj >= Tk) continue;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int c = acc_col(tx, q);
      if (c < dv) a.dV[(bh * Tk + kj) * dv + c] = accV[r][q];
      if (c < d) a.dK[(bh * Tk + kj) * d + c] = accK[r][q] * scale;
    }
  }
}

// Deterministic dQ: one CTA per (64-row query tile, head, key range) loops
// over its key steps of BK keys in a fixed order and writes dQ once. With
// several ranges (a.dq_splits > 1; ranges of a.dq_split_tiles 64-key tiles)
// each writes scale * (its partial dQ) in fp32 to a.dQpart
// [ranges][B*H*Tq][d], and reduce_dq_kernel adds them in range order; a
// range past the causal limit of its query tile returns at once (the
// reduction does not read it). SPLIT: scores from split rows (Q split, K
// whole and split), else by Dot2.
template <int W, int BK, bool SPLIT>
__global__ void __launch_bounds__(NT, 1) dq_kernel(const BwdArgs a) {
  constexpr int LD = W + 4, LDS = BK + 4, NC = BK / 16, NQ = W / 16;
  extern __shared__ __align__(16) float smem_f[];
  float* sQ = smem_f;                            // [BM][LD] Q (split: its coarse parts, then remainders)
  float* sQl = sQ + BM * LD;
  float* sdO = sQ + (SPLIT ? 2 : 1) * BM * LD;   // [BM][LD]
  float* sK = sdO + BM * LD;                     // [BK][LD] (split: then K's coarse parts and remainders)
  float* sKh = sK + BK * LD;
  float* sKl = sKh + BK * LD;
  float* sV = sK + (SPLIT ? 3 : 1) * BK * LD;    // [BK][LD]
  float* sdS = sV + BK * LD;      // [BM][LDS]
  float* sLse = sdS + BM * LDS;   // [BM]
  float* sD = sLse + BM;          // [BM]
  const Problem& p = a.p;
  const int d = p.d, dv = p.dv, Tq = p.Tq, Tk = p.Tk;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int q0 = blockIdx.x * BM;
  const size_t bh = blockIdx.y;
  const float scale = p.scale;
  int n_kt = (Tk + BK - 1) / BK;
  if (p.causal) n_kt = min(n_kt, (q0 + BM - 1) / BK + 1);
  // this CTA's key steps [k0, k1)
  const int steps_per_range = a.dq_split_tiles * (kF32SplitTile / BK);
  const int k0 = a.dq_splits > 1 ? blockIdx.z * steps_per_range : 0;
  const int k1 = a.dq_splits > 1 ? min(n_kt, k0 + steps_per_range) : n_kt;
  if (k0 >= k1 && a.dq_splits > 1) return;

  if constexpr (SPLIT)
    load_split<W, BM>(nullptr, sQ, sQl, LD, a.Q + (bh * Tq + q0) * d, d, Tq - q0);
  else
    load_tile<W>(sQ, LD, a.Q + (bh * Tq + q0) * d, BM, d, Tq - q0);
  load_tile<W>(sdO, LD, a.dO + (bh * Tq + q0) * dv, BM, dv, Tq - q0);
  if (threadIdx.x < BM) {
    const int qi = q0 + threadIdx.x;
    sLse[threadIdx.x] = qi < Tq ? a.LSE[bh * Tq + qi] : -CUDART_INF_F;
    sD[threadIdx.x] = qi < Tq ? a.D[bh * padded_rows(Tq) + qi] : 0.f;
  }
  float acc[4][NQ];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[r][q] = 0.f;
  // split rows: a key step's K and V rows load into registers while the
  // previous step's dQ product runs
  RowRegs<W, BK> kr, vr;
  if constexpr (SPLIT) {
    kr.load(a.K + (bh * Tk + k0 * BK) * d, d, Tk - k0 * BK);
    vr.load(a.V + (bh * Tk + k0 * BK) * dv, dv, Tk - k0 * BK);
  }
  for (int kt = k0; kt < k1; ++kt) {
    const int kv0 = kt * BK;
    __syncthreads();   // the previous step is done with sK, sV, sdS
    if constexpr (SPLIT) {
      kr.split(sK, sKh, sKl, LD);
      vr.store(sV, LD);
    } else {
      load_tile<W>(sK, LD, a.K + (bh * Tk + kv0) * d, BK, d, Tk - kv0);
      load_tile<W>(sV, LD, a.V + (bh * Tk + kv0) * dv, BK, dv, Tk - kv0);
    }
    __syncthreads();
    {
      float sh[4][NC], sl[4][NC], dp[4][NC];
      if constexpr (SPLIT) {
        if (d == dv) {
          split_dot_tile<NC>(sQ, sQl, sK, sKh, sKl, sdO, sV, LD, ty, tx, d, sh, sl, dp);
        } else {
          split_tile<NC, false>(nullptr, sQ, sQl, sK, sKh, sKl, LD, ty, tx, d, sh, sl);
          dot_tile<NC>(sdO, sV, LD, ty, tx, dv, dp);
        }
      } else {
        dot2_tile<NC>(sQ, sK, LD, ty, tx, d, sh, sl);
        dot_tile<NC>(sdO, sV, LD, ty, tx, dv, dp);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = ty + 16 * r, qi = q0 + i;
        const float lse = sLse[i], dd = sD[i];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int kj = kv0 + tx + 16 * c;
          const bool blocked = qi >= Tq || kj >= Tk || (p.causal && kj > qi) || lse == -CUDART_INF_F;
          float pij, dsij;
          p_ds(sh[r][c], sl[r][c], dp[r][c], scale, lse, dd, blocked, pij, dsij);
          sdS[i * LDS + tx + 16 * c] = dsij;
        }
      }
    }
    __syncthreads();
    if constexpr (SPLIT) {
      if (kt + 1 < k1) {
        kr.load(a.K + (bh * Tk + kv0 + BK) * d, d, Tk - kv0 - BK);
        vr.load(a.V + (bh * Tk + kv0 + BK) * dv, dv, Tk - kv0 - BK);
      }
    }
    acc_tile<4, NQ>(sdS, LDS, sK, LD, ty, tx, min(BK, Tk - kv0), acc);
  }
  float* out = a.dq_splits > 1 ? a.dQpart + blockIdx.z * static_cast<size_t>(p.B) * p.H * Tq * d : a.dQ;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int qi = q0 + ty + 16 * r;
    if (qi >= Tq) continue;
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (acc_col(tx, q) < d) out[(bh * Tq + qi) * d + acc_col(tx, q)] = acc[r][q] * scale;
  }
}

// dQ = the sum of the dQ kernel's partials (already scaled) in range order,
// over the ranges that hold key tiles of the row's query tile: one thread per
// element (any d).
__global__ void __launch_bounds__(256) reduce_dq_kernel(const float* __restrict__ part, float* __restrict__ out,
                                                        long long rows, int Tq, int d, int n_ranges,
                                                        int range_tiles, int n_k_tiles, int causal) {
  const long long n = rows * d;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int qt = static_cast<int>((i / d) % Tq) / kF32SplitTile;
    const int nt = causal ? min(qt + 1, n_k_tiles) : n_k_tiles;
    const int ns = min(n_ranges, (nt + range_tiles - 1) / range_tiles);
    float acc = 0.f;
    for (int s = 0; s < ns; ++s) acc += part[static_cast<long long>(s) * n + i];
    out[i] = acc;
  }
}

// Queries per step of the dK/dV kernel and keys per step of the dQ kernel:
// 32 from W = 128 on, 64 at W = 64, so that the split tiles fit in shared
// memory (one CTA per SM).
template <int W>
constexpr int dkdv_rows() { return W >= 128 ? 32 : 64; }
template <int W>
constexpr int dq_rows() { return W >= 128 ? 32 : 64; }

template <int W, bool SPLIT>
constexpr size_t dkdv_smem_of() {
  constexpr int BQ = dkdv_rows<W>();
  // (split rows: one more [BM][W + 4] tile, the whole K for the atomic dQ product)
  return sizeof(float) * ((SPLIT ? 4 : 2) * BM * (W + 4) + (SPLIT ? 4 : 2) * BQ * (W + 4) + 2 * BM * (BQ + 4) + 2 * BQ +
                          BQ * (BM + 4));
}
// split rows wherever their tiles fit
template <int W>
constexpr bool dkdv_split() { return dkdv_smem_of<W, true>() <= kSmemMax; }
template <int W>
constexpr size_t dkdv_smem() { return dkdv_smem_of<W, dkdv_split<W>()>(); }

template <int W, bool SPLIT>
constexpr size_t dq_smem_of() {
  constexpr int BK = dq_rows<W>();
  return sizeof(float) * ((SPLIT ? 3 : 2) * BM * (W + 4) + (SPLIT ? 4 : 2) * BK * (W + 4) + BM * (BK + 4) + 2 * BM);
}
template <int W>
constexpr bool dq_split() { return dq_smem_of<W, true>() <= kSmemMax; }
template <int W>
constexpr size_t dq_smem() { return dq_smem_of<W, dq_split<W>()>(); }

template <int W>
cudaError_t bwd_launch(const LaunchBwd& la, const BwdArgs& b, bool kv, bool q, bool red) {
  constexpr int RQ = dkdv_rows<W>(), RK = dq_rows<W>();
  constexpr size_t s1 = dkdv_smem<W>(), s2 = dq_smem<W>();
  static_assert(s1 <= kSmemMax && s2 <= kSmemMax, "shared memory");
  const Problem& p = la.p;
  cudaError_t e;
  if (kv && p.Tk > 0) {
    constexpr bool SP = dkdv_split<W>();
    e = cudaFuncSetAttribute(dkdv_kernel<W, RQ, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(s1));
    if (e != cudaSuccess) return e;
    dim3 g1((p.Tk + BM - 1) / BM, p.B * p.H);
    dkdv_kernel<W, RQ, SP><<<g1, NT, s1, la.stream>>>(b, !la.deterministic ? 1 : f32_fused_dq(p.B, p.H, p.Tq, p.Tk, p.d) ? 2 : 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (q) {
    constexpr bool SP = dq_split<W>();
    e = cudaFuncSetAttribute(dq_kernel<W, RK, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(s2));
    if (e != cudaSuccess) return e;
    dim3 g2((p.Tq + BM - 1) / BM, p.B * p.H, b.dq_splits > 1 ? b.dq_splits : 1);
    dq_kernel<W, RK, SP><<<g2, NT, s2, la.stream>>>(b);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (red && b.dq_splits > 1) {
    const long long rows = static_cast<long long>(p.B) * p.H * p.Tq;
    reduce_dq_kernel<<<la.num_sms * 8, 256, 0, la.stream>>>(
        b.dQpart, b.dQ, rows, p.Tq, p.d, b.dq_splits, b.dq_split_tiles,
        (p.Tk + kF32SplitTile - 1) / kF32SplitTile, p.causal);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace simt

size_t fwd_f32_smem_bytes(int block_n, int d, int dv) {
  using namespace simt;
  const int W = tile_width(d, dv);
  switch (block_n) {
    case 32: return W == 64 ? fwd_smem<64, 32>() : W == 128 ? fwd_smem<128, 32>() : fwd_smem<256, 32>();
    case 128: return W == 64 ? fwd_smem<64, 128>() : W == 128 ? fwd_smem<128, 128>() : fwd_smem<256, 128>();
    default: return W == 64 ? fwd_smem<64, 64>() : W == 128 ? fwd_smem<128, 64>() : fwd_smem<256, 64>();
  }
}

cudaError_t launch_fwd_f32(const LaunchFwd& a) {
  using namespace simt;
  static_assert(BM == kF32SplitTile, "key ranges count 64-row query tiles and 64-key tiles");
  const int W = tile_width(a.p.d, a.p.dv);
  if (a.n_splits > 1 && a.block_n != kF32SplitTile) return cudaErrorInvalidValue;
  switch (a.block_n) {
    case 32: return W == 64 ? fwd_launch<64, 32>(a) : W == 128 ? fwd_launch<128, 32>(a) : fwd_launch<256, 32>(a);
    case 128:
      // a 128-key tile of rows wider than 128 columns does not fit in shared
      // memory (the host refuses it before the launch)
      return W == 64 ? fwd_launch<64, 128>(a) : W == 128 ? fwd_launch<128, 128>(a) : cudaErrorInvalidValue;
    default: return W == 64 ? fwd_launch<64, 64>(a) : W == 128 ? fwd_launch<128, 64>(a) : fwd_launch<256, 64>(a);
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
  // (no dQ kernel where the dK/dV kernel writes the key tiles' partials)
  const bool q = a.deterministic && !f32_fused_dq(p.B, p.H, p.Tq, p.Tk, p.d) && (a.phase == 0 || a.phase == 2 || a.phase == 5);
  // the sum of the range partials (phase 3, as for bf16)
  const bool red = a.deterministic && a.dq_splits > 1 && (a.phase == 0 || a.phase == 3);
  if (!kv && !q && !red) return cudaSuccess;
  if ((q || red || (kv && a.deterministic)) && a.dq_splits > 1 && a.dQpart == nullptr) return cudaErrorInvalidValue;
  simt::BwdArgs b{static_cast<const float*>(a.Q), static_cast<const float*>(a.K), static_cast<const float*>(a.V),
                  static_cast<const float*>(a.dO), a.LSE, a.D, static_cast<float*>(a.dQ),
                  static_cast<float*>(a.dK), static_cast<float*>(a.dV), p,
                  a.deterministic ? a.dq_splits : 1, a.dq_split_tiles, a.dQpart};
  const int W = simt::tile_width(p.d, p.dv);
  return W == 64 ? simt::bwd_launch<64>(a, b, kv, q, red)
                 : W == 128 ? simt::bwd_launch<128>(a, b, kv, q, red) : simt::bwd_launch<256>(a, b, kv, q, red);
}

}  // namespace attn
