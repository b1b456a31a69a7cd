/*
 * attn.h -- C ABI of the exact tiled softmax attention library (libattn.so).
 *
 * Exact scaled-dot-product softmax attention, forward and backward, computed
 * one key tile at a time with an online softmax, so the Tq x Tk score matrix
 * is never stored. Kernels are written for NVIDIA sm_103a (GB300).
 *
 * Definitions (sources are the pages this library restates):
 *   S   = scale * Q K^T, with S_ij = -inf where the mask blocks key j for
 *         query i. causal = 1 blocks j > i with global row indices
 *         ("Tiled attention with an online softmax", section "Task").
 *   O   = softmax(S) V                ("The Hidden Recurrence in Softmax
 *         Attention", section "Standard Attention / Forward Pass";
 *         "attention_backprop", section "Forward Pass")
 *   LSE = log sum_j exp(S_ij)         (natural log; the page's m_i + log l_i)
 *   D   = rowsum(dO o O)
 *   dV  = P^T dO,  dS = P o (dO V^T - D),  dQ = scale * dS K,
 *   dK  = scale * dS^T Q              ("attention_backprop", sections
 *         "Gradient of V and P", "Gradient of S", "Gradient of Q and K";
 *         the factor scale comes from S = scale * Q K^T)
 *
 * Layout: every tensor is a contiguous row-major device array.
 *   Q [B,H,Tq,d]  K [B,H,Tk,d]  V [B,H,Tk,dv]  O, dO [B,H,Tq,dv]
 *   dQ [B,H,Tq,d] dK [B,H,Tk,d] dV [B,H,Tk,dv] LSE, D [B,H,Tq] (fp32)
 * Q, K, V, O, dO, dQ, dK, dV use the element type `dtype`; LSE is always fp32.
 *
 * Ownership: the caller allocates and owns every buffer, including the
 * backward workspace. The library never allocates device memory in these
 * calls and never writes its inputs. Outputs must not overlap inputs.
 *
 * Asynchrony: every call validates its arguments on the host, then enqueues
 * kernels on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 * stream) and returns without synchronising. A nonzero status from the host
 * checks means nothing was enqueued.
 *
 * Supported shapes:
 *   ATTN_F32 : 1 <= d, dv <= 256, any B, H, Tq, Tk >= 0 (attn_fwd_f32_blocked
 *              with block_n = 128 returns ATTN_ERR_UNSUPPORTED when its key
 *              tile does not fit in shared memory: d or dv above 128)
 *   ATTN_BF16: forward (attn_fwd, attn_fwd_splitkv): d and dv multiples
 *              of 8 from 8 to 256, independently (the page's task takes V
 *              with its own head dimension); a width below 64, 128 or 256
 *              runs on the next of those tile widths with zero columns, so
 *              64, 128 and 256 are the efficient sizes. Backward (attn_bwd):
 *              d and dv multiples of 8 up to 256, independently. The
 *              kernels take d, dv in {64, 128}, and d = 256 with dv in {64,
 *              128, 256}; other widths run on zero-padded copies of the
 *              inputs held in the workspace (rows wider than 128 on either
 *              side pad d to 256), and attn_bwd_phase takes only the
 *              kernels' own widths. Any B, H, Tq, Tk >= 0.
 * Zero-sized problems are valid: Tk == 0 gives O = 0 and LSE = -inf (a row
 * with no allowed key), and empty gradients are written as zeros.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, negative size, non-finite or non-positive scale, overlap */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement (e.g. bf16 with d = 96) */
  ATTN_ERR_MISALIGNED = 3,   /* a pointer breaks the alignment rule of its dtype (bf16: 16 B, f32: 4 B) */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed; see attn_last_cuda_error() */
  ATTN_ERR_TIMEOUT = 5,      /* a kernel's bounded pipeline wait gave up (reported by attn_device_status) */
  ATTN_ERR_WORKSPACE = 6     /* workspace missing, too small or not 256-byte aligned */
} attn_status_t;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/*
 * Forward pass: O and LSE from Q, K, V.
 * Restates flash_attention of "Tiled attention with an online softmax"
 * (sections "Task", "Input and output") for a batch of heads: returns the
 * attention output and the log-sum-exp of each query row. `scale` multiplies
 * Q K^T (the page uses 1/sqrt(d); pass that for the same result) and must be
 * finite and > 0. `causal` is 0 (no mask) or 1.
 * Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_MISALIGNED,
 * ATTN_ERR_CUDA (launch failure).
 */
ATTN_API attn_status_t attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Tq,
                       int Tk, int d, int dv, float scale, int causal, attn_dtype_t dtype, void* stream);

/*
 * Forward pass of the fp32 path with an explicit key-tile size (keys per
 * online-softmax step): block_n in {32, 64, 128}. The result must not depend
 * on it ("Tiled attention with an online softmax", section "Constraints":
 * equal to standard attention for every block size). attn_fwd uses 64.
 * Same arguments and errors as attn_fwd with dtype ATTN_F32.
 */
ATTN_API attn_status_t attn_fwd_f32_blocked(const float* Q, const float* K, const float* V, float* O, float* LSE, int B,
                                   int H, int Tq, int Tk, int d, int dv, float scale, int causal, int block_n,
                                   void* stream);

/*
 * Split-KV forward for problems with few query tiles per SM (small B*H*Tq,
 * long Tk): the key tiles of every query-tile unit (bf16: a pair of 128-row
 * query tiles, one tile for d = 256, 128-key tiles; fp32: one 64-row query
 * tile, 64-key tiles) are divided into S contiguous ranges ("splits") that
 * run as separate work units; each
 * writes its partial softmax state for its keys (O_s = A_s / l_s and LSE_s,
 * fp32) to `workspace`, and a merge kernel combines the splits with the
 * associative rescale of the running max, sum and accumulator ("The Hidden
 * Recurrence in Softmax Attention", section "Chunk-wise Mode with Online
 * Softmax Re-scale": chunk states rescaled to a common maximum and added):
 *   M = max_s LSE_s, w_s = exp(LSE_s - M), O = sum_s w_s O_s / sum_s w_s,
 *   LSE = M + log sum_s w_s.
 * Same inputs, outputs, layout and mask as attn_fwd; O and LSE agree with
 * attn_fwd up to fp32 rounding order. num_splits = 0 picks S from the
 * current device's SM count: the smallest S whose time (the waves of units
 * x S work units over the SMs, times the key tiles of a split) is within 5 %
 * of the best, at least two key tiles per split; a bf16 problem with at
 * least as many units as SMs keeps S = 1. num_splits >= 1 asks for that
 * many, clamped to the number of key tiles and 64. S = 1 is attn_fwd itself (no workspace). `workspace`
 * (256-byte aligned, at least attn_fwd_splitkv_workspace_size bytes, not
 * overlapping any other argument; may be NULL when that is 0) holds Opart
 * [S][B*H*Tq][dv] fp32 then LSEpart [S][B*H*Tq] (fp32 for bf16 problems;
 * fp64 for fp32 ones, whose merge weights exp(LSE_s - max) must keep fp32
 * accuracy at logits in the thousands); else ATTN_ERR_WORKSPACE. Other
 * errors as attn_fwd; asynchronous on `stream`.
 */
ATTN_API attn_status_t attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                        int H, int Tq, int Tk, int d, int dv, float scale, int causal,
                                        attn_dtype_t dtype, int num_splits, void* workspace,
                                        size_t workspace_bytes, void* stream);

/*
 * The number of splits S attn_fwd_splitkv uses for these arguments (>= 1;
 * num_splits = 0 consults the current device's SM count), or -1 for invalid
 * arguments.
 */
ATTN_API int attn_fwd_splitkv_splits(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype,
                                     int num_splits);

/*
 * Bytes of workspace attn_fwd_splitkv needs (0 when S = 1 or the arguments
 * are invalid).
 */
ATTN_API size_t attn_fwd_splitkv_workspace_size(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype,
                                                int num_splits);

/*
 * Bytes of device workspace attn_bwd needs for this problem (0 is possible).
 * Holds -LSE * log2(e) and D = rowsum(dO o O), each [B*H, Tq_pad] fp32 with
 * Tq_pad = Tq rounded up to a multiple of 128, and, for bf16 with d <= 128
 * and deterministic == 0, the fp32 dQ accumulator [B,H,Tq,d], or, with
 * deterministic == 1 and S = attn_bwd_dq_splits(...) > 1 (either dtype), S
 * fp32 partial dQ arrays [S][B,H,Tq,d], and, for bf16 with d <= 128, 256 bytes of counters
 * through which the dQ and dK/dV kernels hand out their work units at run
 * time (reset by each call); each part starts on a 256-byte boundary. For bf16
 * widths other than 64 and 128 it first holds zero-padded bf16 copies of Q,
 * K, V, O, dO and of the three gradients, in rows of the next tile width (64,
 * 128 or 256 columns), then the workspace above for the padded widths; the
 * padded problem's dQ splits are the ones attn_bwd_dq_splits reports.
 * Returns 0 for invalid arguments as well.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype,
                               int deterministic);

/*
 * Number of key splits S the deterministic backward uses for dQ (1 when it
 * does not split; -1 for invalid arguments). Each query tile's keys are cut
 * into S ranges whose partial dQ go to the workspace and are then added in
 * split order, so the result stays bitwise reproducible. bf16: the dQ kernel
 * runs one unit per 128-row query tile; when there are fewer such units than
 * 76 (half of a GB300's 152 SMs) and at least 8 key tiles, S ranges of at
 * least 4 key tiles each, at most 152 units in all, S <= 64. fp32: with at
 * most 1 GiB of partials (S x B*H*Tq*d*4 bytes for S the number of 64-key
 * tiles), every key tile is a range of its own (S = the number of key tiles):
 * the dK/dV kernel writes each key tile's partial dQ (with one key tile, dQ
 * itself) and no separate dQ pass runs. Otherwise the dQ pass runs one unit
 * per 64-row query tile over ranges of 64-key tiles; S is the smallest count
 * whose time (the waves of units x S on 152 SMs, times the key tiles of a
 * range) is within 5 % of the best, at least two key tiles per range, S <=
 * 64. Rules of the shapes only, so that the workspace size needs no device:
 * the 152 is GB300's SM count, and on a device with another SM count the
 * split stays correct but fills the SMs less evenly.
 */
ATTN_API int attn_bwd_dq_splits(int B, int H, int Tq, int Tk, int d, int dv, attn_dtype_t dtype,
                                int deterministic);

/*
 * Backward pass: dQ, dK, dV from Q, K, V, the forward's O and LSE, and dO.
 * Recomputes P tile by tile from LSE instead of storing it ("The Hidden
 * Recurrence in Softmax Attention", section "Flash Attention Backward Pass":
 * store the row statistics, recompute the attention matrix per tile), forms
 * D = rowsum(dO o O), and accumulates the per-tile gradient terms of
 * "attention_backprop" (sections "Gradient of V and P" through "Gradient of
 * Q and K"). `O` and `LSE` must be the outputs of attn_fwd on the same
 * inputs, scale and mask. deterministic = 1 sums the key tiles' shares of
 * dQ in a fixed order (bitwise reproducible): bf16 in a separate dQ pass;
 * fp32 from one partial per 64-key tile that the dK/dV pass writes, added in
 * key-tile order, or, above 1 GiB of such partials, in a separate dQ pass
 * (attn_bwd_dq_splits). 0 adds each key tile's share with fp32 atomics. For
 * bf16 rows of 256 columns both
 * values run the fixed-order pass: there a dQ kernel, a dV kernel and a dK
 * kernel each hold one 256-column accumulator (tensor memory has room for
 * one next to the score tiles), all bitwise reproducible. `workspace` (256-byte aligned, at least
 * attn_bwd_workspace_size bytes; may be NULL when that is 0) is scratch
 * owned by the caller and overwritten.
 * Errors: as attn_fwd, plus ATTN_ERR_WORKSPACE.
 */
ATTN_API attn_status_t attn_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                       const void* dO, void* dQ, void* dK, void* dV, int B, int H, int Tq, int Tk, int d, int dv,
                       float scale, int causal, attn_dtype_t dtype, int deterministic, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * The backward split into its launch groups, for measurement: the same
 * arguments as attn_bwd plus `phase`:
 *   1  preprocess: D = rowsum(dO o O) and -LSE * log2(e) (and zeroing of the
 *      fp32 dQ accumulator when deterministic == 0); a no-op for bf16 with
 *      deterministic == 1 and for bf16 rows wider than 128 columns, where
 *      the dQ kernel forms D itself
 *   2  main kernels: phases 5 and 4 in this order
 *   3  dQ conversion from the fp32 accumulator (bf16 with deterministic
 *      == 0), or the in-order sum of the split dQ partials (bf16 with
 *      deterministic == 1 and attn_bwd_dq_splits(...) > 1); a no-op otherwise
 *   4  the dK/dV kernel alone (with deterministic == 0 it also accumulates dQ;
 *      bf16 rows wider than 128 columns: the dV and the dK kernel)
 *   5  the separate dQ kernel alone (deterministic == 1, or bf16 rows wider
 *      than 128 columns; a no-op otherwise); for bf16 it also writes the D
 *      and -LSE * log2(e) phase 4 reads
 *   6  in place of phase 5, the same dQ pass on CTA pairs: two 128-row query
 *      tiles per cluster of two CTAs, each tensor-core product computed for
 *      both at once with the K and V operands split between the two SMs
 *      (bf16, d = 128, deterministic == 1 only, else ATTN_ERR_UNSUPPORTED).
 *      Same results within rounding; attn_bwd does not use it (on GB300 at
 *      B=2 H=16 T=8192 it is slower than phase 5).
 * Calling phases 1, 2, 3 (or 1, 5, 4, 3, or 1, 6, 4, 3) in order on one
 * stream equals one attn_bwd call; phase 0 is attn_bwd itself. Other values
 * give ATTN_ERR_INVALID_ARG.
 */
ATTN_API attn_status_t attn_bwd_phase(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                                      const void* dO, void* dQ, void* dK, void* dV, int B, int H, int Tq, int Tk,
                                      int d, int dv, float scale, int causal, attn_dtype_t dtype, int deterministic,
                                      void* workspace, size_t workspace_bytes, int phase, void* stream);

/*
 * Size of the static scratch buffer behind attn_bwd_noalloc (64 MiB). A
 * device holds a buffer of this size from the moment the library's code is
 * loaded on it until the process exits. With CUDA's lazy module loading (the
 * default since CUDA 12.2) that moment is the first attn_bwd_noalloc call on
 * the device; with eager loading (CUDA_MODULE_LOADING=EAGER) it is the
 * library's first use of the device.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * attn_bwd for callers that cannot allocate device memory: a host without
 * its own CUDA allocator or memory pool, a plug-in that may not grow the
 * process's device footprint, or a loop where a cudaMalloc (which can
 * synchronise the device) is not acceptable. The pages have no counterpart
 * to this call; it exists only for such callers.
 *
 * Arguments, layout and results are those of attn_bwd, without the workspace
 * arguments: the workspace lives in a static device buffer of
 * ATTN_NOALLOC_SCRATCH_BYTES inside the library (static device data of the
 * library's module, not a cudaMalloc). The call calls no cudaMalloc,
 * cudaFree or other allocating routine. Problems whose attn_bwd_workspace_size
 * exceeds that size are rejected with ATTN_ERR_WORKSPACE before anything is
 * enqueued (for bf16 with deterministic == 0 the need is about
 * B*H*Tq*(d+2)*4 bytes; deterministic == 1 or fp32 needs about B*H*Tq*8).
 *
 * The first call on a device (with that device current) looks up the
 * buffer's device address, and under lazy module loading that lookup is
 * also what reserves the 64 MiB on the device, so it can fail with
 * ATTN_ERR_CUDA (for example while the device's memory is full). Only a
 * successful lookup is kept: after a failure the next call tries again.
 * Make the first call on each device before any stream capture begins.
 * All calls on a device share the one buffer and leave their data in it; each call overwrites everything it reads back (D, and the fp32
 * dQ accumulator, which it zeroes first). Calls whose kernels can overlap on
 * the GPU (different streams without ordering, or several host threads) race
 * on the buffer and corrupt each other's gradients: order them on one stream.
 */
ATTN_API attn_status_t attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                        const float* LSE, const void* dO, void* dQ, void* dK, void* dV, int B,
                                        int H, int Tq, int Tk, int d, int dv, float scale, int causal,
                                        attn_dtype_t dtype, int deterministic, void* stream);

/*
 * One step of the online softmax, on the device: for each of the n query
 * rows, fold one block of bs keys into the running state ("Tiled attention
 * with an online softmax", section "Task": the online_softmax_step of the
 * page; "The Hidden Recurrence in Softmax Attention", section "Chunk-wise
 * Mode with Online Softmax Re-scale"):
 *   m' = max(m, max_j s_ij), with 0 used for m' inside the exponentials when
 *        m' = -inf (a row with no allowed key so far)
 *   l' = exp(m - m') l + sum_j exp(s_ij - m')
 *   acc' = exp(m - m') acc + sum_j exp(s_ij - m') v_j
 * m, l [n] and acc [n, dv] (row-major) are fp32 device buffers updated in
 * place; a fresh row is m = -inf, l = 0, acc = 0, and acc / l is its
 * attention output once every block has been folded in. scores [n, bs] fp32
 * (-inf marks a blocked key) and v_block [bs, dv] fp32 are read only. The
 * arithmetic runs in fp64. n, bs >= 0 and 1 <= dv <= 512; buffers 4-byte
 * aligned, the three outputs disjoint from each other and from the inputs,
 * else ATTN_ERR_INVALID_ARG / ATTN_ERR_MISALIGNED before any launch.
 * Asynchronous on `stream`.
 */
ATTN_API attn_status_t attn_online_softmax_step(float* m, float* l, float* acc, const float* scores,
                                                const float* v_block, int n, int bs, int dv, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word that
 * the kernels set when a bounded wait gives up (ATTN_ERR_TIMEOUT) or a launch
 * precondition fails on the device (ATTN_ERR_CUDA). ATTN_OK otherwise.
 * Intended for tests and debugging; it blocks the host.
 */
ATTN_API attn_status_t attn_device_status(void* stream);

/*
 * Test hook for the bounded wait itself: launches one CTA that waits on an
 * mbarrier nobody arrives at, with a limit of `limit_ms` milliseconds
 * (1..5000). The kernel gives up, records ATTN_ERR_TIMEOUT in the device
 * status word and exits normally; the context stays usable. Returns the
 * launch status; read the outcome with attn_device_status().
 */
ATTN_API attn_status_t attn_selftest_wait_timeout(int limit_ms, void* stream);

/* Human-readable text for a status code (static storage). */
ATTN_API const char* attn_strerror(attn_status_t status);

/* The cudaError_t (as int) of the last ATTN_ERR_CUDA on this thread, else 0. */
ATTN_API int attn_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
