// specv_verify_chain_noalloc: chain verification with a built-in scratch
// buffer instead of a caller-owned workspace.  The pages describe no such
// call; it exists for callers that cannot hand the library device memory:
//  - code that runs where allocating would deadlock or recurse, such as a
//    callback of a caching device allocator or memory pool;
//  - serving processes that carve all free HBM into weights and KV-cache
//    blocks at start-up and forbid device allocation afterwards;
//  - plain C hosts with no device allocator of their own.
// Every launch and kernel is that of specv_verify_chain; only where the
// scratch lives differs.
#include <cuda_runtime.h>

#include "host_common.h"
#include "specv.h"

namespace {

// Module-scope scratch, one copy per device (a __device__ variable is
// instantiated in every device context that loads this module).
static __device__ __align__(256) unsigned char g_verify_scratch[SPECV_NOALLOC_SCRATCH_BYTES];

// Device address of the current device's copy of g_verify_scratch in the
// current context.  The first call on a device loads the library's device
// module there (the set-up step); after that cudaGetSymbolAddress is a host
// lookup.  It runs on every call rather than being cached: after
// cudaDeviceReset, or in another context on the same device, the buffer has
// another address, and a stale one would send the kernels to unmapped memory.
specv_status scratch_for_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();                 // leave no pending error behind
    return SPECV_ERR_CUDA;
  }
  if (!specv::aligned_to(p, 256)) return SPECV_ERR_CUDA;
  *out = p;
  return SPECV_OK;
}

}  // namespace

extern "C" specv_status specv_verify_chain_noalloc(const void* target_logits, const void* draft_logits,
                                                   specv_dtype dtype, const int32_t* draft_tokens,
                                                   const int32_t* lengths, const float* uniforms, int R, int gamma,
                                                   int V, float temperature, int32_t* accepted_len,
                                                   int32_t* out_token, float* c_star, void* stream) {
  // An empty batch validates its arguments and enqueues nothing.
  if (R == 0)
    return specv_verify_chain(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R, gamma, V,
                              temperature, accepted_len, out_token, c_star, nullptr, 0, stream);
  // Host-only size check first: a shape that does not fit touches no device.
  const size_t need = specv_verify_chain_workspace_size(R, gamma, V, dtype);
  if (need == 0) return SPECV_ERR_INVALID_ARG;
  if (need > SPECV_NOALLOC_SCRATCH_BYTES) return SPECV_ERR_SCRATCH_LIMIT;
  // A device without an sm_103a image reports SPECV_ERR_UNSUPPORTED before
  // the symbol lookup, which would fail there.
  specv_status s = specv::check_device();
  if (s != SPECV_OK) return s;
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != SPECV_OK) return s;
  // The only word that must start at zero, the device error word in the first
  // 256 bytes, is cleared by the first kernel of every call.
  return specv_verify_chain(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R, gamma, V,
                            temperature, accepted_len, out_token, c_star, scratch, SPECV_NOALLOC_SCRATCH_BYTES,
                            stream);
}
