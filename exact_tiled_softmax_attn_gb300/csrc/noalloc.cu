// attn_bwd_noalloc: the backward pass with its scratch memory in a static
// device buffer of this library, for callers that cannot allocate device
// memory themselves.
//
// attn_bwd needs a caller-provided workspace (D = rowsum(dO o O) and, for
// bf16 with fp32 dQ accumulation, a [B,H,Tq,d] fp32 accumulator). Some hosts
// have no way to get one: a plain C program that owns no CUDA allocator or
// memory pool, a plug-in that is handed device tensors but is not allowed to
// grow the process's device footprint at run time, or a latency-critical
// loop where a cudaMalloc (which can synchronise the device) is not
// acceptable. This entry point takes the same inputs and outputs as attn_bwd
// and uses kNoAllocScratchBytes of scratch that every device holds from the
// moment it loads the library until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "attn.h"

namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;

// The scratch itself. In host code this name is only a stand-in for the
// device object; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_slots_mu;
void* g_slots[kMaxDevices];   // device address of the scratch per device, once looked up

// Device address of the scratch on the current device. Only a successful
// lookup is kept: with lazy module loading the first lookup on a device is
// also what loads this file's module and reserves the buffer there, and it
// can fail (for example while the device's memory is full); the next call
// then tries again instead of failing for good.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_slots_mu);
  if (g_slots[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();   // leave no sticky record of the failed lookup
      return e;
    }
    g_slots[dev] = p;
  }
  *out = g_slots[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace attn

extern "C" attn_status_t attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                          const float* LSE, const void* dO, void* dQ, void* dK, void* dV, int B,
                                          int H, int Tq, int Tk, int d, int dv, float scale, int causal,
                                          attn_dtype_t dtype, int deterministic, void* stream) {
  // Same argument checks as attn_bwd; a zero size means "invalid" there too.
  const size_t need = attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, dtype, deterministic);
  if (need > attn::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const cudaError_t e = attn::scratch_address(&scratch);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  // attn_bwd writes D (and, for padded bf16 widths, the padded copies of its
  // inputs) in full and zeroes the fp32 dQ accumulator before it accumulates,
  // so whatever an earlier call left in the scratch is not read.
  return attn_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, Tq, Tk, d, dv, scale, causal, dtype, deterministic,
                  scratch, attn::kNoAllocScratchBytes, stream);
}
