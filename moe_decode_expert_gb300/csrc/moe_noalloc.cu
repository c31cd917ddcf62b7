// moe_noalloc.cu — a T = 1 decode entry point for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc or to hand the library a
// workspace: code running under an allocator that forbids new device
// allocations (a fixed memory pool reserved at start-up), plugins that only
// receive input and output pointers from a host framework, or hosts that
// capture work while allocation is disallowed.  For them this file keeps the
// decode kernel's scratch (the control block and the exchange words the CTAs
// pass each other) in a file-scope device array, so the call needs nothing
// beyond the tensors themselves.
//
// The array is fixed at kNoAllocScratchBytes and stays resident on every GPU
// that loads the library until the process exits.  All calls share it, so
// two calls that can overlap on the GPU (different streams, or the same
// array used from two threads) race and must be serialised by the caller.
// Each call clears the part of the array it uses before its kernel runs, so
// no state carries over from the previous call, except the device status
// word: a device-side error (a wait that ran out) stays recorded until
// moe_query_status(NULL, stream) reads and clears it.

#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (host code only sees a host-side stand-in for the symbol).
static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64];

moe_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(MOE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return set_error(MOE_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_decode_forward_noalloc(const moe_cfg_t* cfg, const void* x, const void* router_w,
                                                   const void* w13, const void* w2, const void* shared_w13,
                                                   const void* shared_w2, const void* shared_gate_w,
                                                   moe_topk_t topk, void* out, void* stream) {
  if (!cfg) return set_error(MOE_ERR_INVALID_ARG, "cfg is NULL");
  const size_t need = moe_workspace_bytes(cfg, 1);
  if (need == 0) return set_error(MOE_ERR_INVALID_ARG, "invalid cfg");
  if (need > kNoAllocScratchBytes)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "moe_decode_forward_noalloc: this cfg needs %zu bytes of scratch, the built-in "
                     "array holds %zu (use moe_decode_forward with a workspace)",
                     need, kNoAllocScratchBytes);
  // Every argument is checked before anything is enqueued, so a rejected call
  // leaves the shared array (and any call still running on it) untouched.
  if (moe_status_t s = check_block(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, topk, out))
    return s;
  void* scratch = nullptr;
  if (moe_status_t s = noalloc_scratch(&scratch)) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Start every call from a zeroed control block and zeroed exchange words,
  // except the first two words (device status, detail): an error recorded by
  // an earlier call stays there until moe_query_status(NULL, ...) reads it.
  constexpr size_t kKeep = 2 * sizeof(uint32_t);
  if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + kKeep, 0, need - kKeep, st) != cudaSuccess)
    return check_launch("cudaMemsetAsync(scratch)");
  return moe_decode_forward(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, topk, out,
                            scratch, need, stream);
}
