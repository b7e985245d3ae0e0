// Fixed device scratch for ccv_bwd_noalloc (see include/ccv.h).
//
// The backward pass needs a scratch buffer for its FP32 parameter-gradient
// partials.  ccv_bwd takes it from the caller; ccv_bwd_noalloc uses this
// file-scope array instead, so that a caller which cannot allocate device
// memory at the call site still gets dweight and dbias.  The array is part of
// the library's device image: it exists once per device the library is loaded
// on, from module load on, and nothing here allocates.
#include <cuda_runtime.h>

#include "ccv_internal.h"

namespace ccv {
namespace {

constexpr size_t kNoallocScratchBytes = size_t{16} << 20;  // 16 MiB

// Partial sums written and then read by one ccv_bwd_noalloc call; no slot has
// to start at zero (the gradient kernel writes each slot it uses before the
// reduction kernel reads it).
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

}  // namespace

size_t noalloc_scratch_bytes() { return kNoallocScratchBytes; }

// Address of the scratch on the CURRENT device.
cudaError_t noalloc_scratch_address(void** ptr) {
  return cudaGetSymbolAddress(ptr, g_noalloc_scratch);
}

}  // namespace ccv
