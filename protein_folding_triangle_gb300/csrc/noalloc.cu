// Allocation-free entry point of the backward: the same five kernels as
// tri_attn_bwd (preprocess, bias transpose, main, dQ reduce, dbias reduce),
// with their scratch memory in a file-scope device array instead of a
// caller-provided workspace.  Declared in include/triattn.h.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "triattn.h"

namespace {

constexpr size_t kScratchBytes = TRIATTN_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code this name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

}  // namespace

extern "C" triattn_status tri_attn_bwd_noalloc(const triattn_shape* shape, const void* q, const void* k,
                                               const void* v, const void* bias, const void* mask, const void* o,
                                               const void* o_resid, const float* lse, const void* dO, void* dq,
                                               void* dk, void* dv, void* dbias, void* stream) {
  const size_t need = triattn_bwd_workspace_bytes(shape);
  if (need == 0) {
    // invalid shape: let the regular entry point report which check failed
    return tri_attn_bwd(shape, q, k, v, bias, mask, o, o_resid, lse, dO, dq, dk, dv, dbias, nullptr, 0, stream);
  }
  if (need > kScratchBytes) return TRIATTN_ERR_WORKSPACE;
  // The array's device address on the current device, looked up on every
  // call: the lookup allocates nothing and is cheap, and an address kept
  // from an earlier call would be stale after a device reset.
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr) return TRIATTN_ERR_CUDA;
  return tri_attn_bwd(shape, q, k, v, bias, mask, o, o_resid, lse, dO, dq, dk, dv, dbias, scratch, kScratchBytes,
                      stream);
}
