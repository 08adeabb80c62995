// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.  Some callers have no way to get a workspace: code running where
// cudaMalloc is not allowed or not wanted (inside an allocator hook, a
// plug-in that must not touch the process's memory pool, a pre-allocated
// real-time pipeline).  For them the library keeps its own scratch: one
// file-scope device array, FA_NOALLOC_SCRATCH_BYTES long, that exists on every
// GPU that loads this library until the process exits.  The call then runs
// exactly the kernels of fa_bwd with that array as the workspace.
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_context.h"

namespace fa {
namespace {

// The shared scratch.  On the host this name is only a stand-in for the
// device symbol: host code must pass the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Its device address, looked up with cudaGetSymbolAddress on the first call
// in each context (with that context's device current) and cached by the
// context's unique ID: an address from one context is not valid in another,
// nor in a primary context created again after a reset.
PerContextAddress g_noalloc_addr;

int noalloc_scratch(void** out) {
  return g_noalloc_addr.get(out, [](void** p) { return cudaGetSymbolAddress(p, g_noalloc_scratch); }) == 0
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                              float scale, int causal, cudaStream_t stream) {
  // Validate every argument exactly as fa_bwd does before looking at the size:
  // fa_bwd checks sizes, scale, mask flag and pointers ahead of its workspace
  // and, given none, returns without touching the device.  FA_ERR_WORKSPACE
  // from this call therefore means every other argument is valid.
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  const int arg = fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, nullptr,
                         need ? need : 1, nullptr);
  if (arg != FA_ERR_WORKSPACE) return arg;
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = fa::noalloc_scratch(&scratch);
  if (st != FA_OK) return st;
  // fa_bwd's first kernel rewrites every part of the workspace that must start
  // at a known value (it zeroes the dQ accumulator), so the contents left by
  // an earlier call do not matter.
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch, FA_NOALLOC_SCRATCH_BYTES,
                stream);
}
