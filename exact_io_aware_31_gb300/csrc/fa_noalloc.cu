// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.  Some callers have no way to get a workspace: code running where
// cudaMalloc is not allowed or not wanted (inside an allocator hook, a
// plug-in that must not touch the process's memory pool, a pre-allocated
// real-time pipeline).  For them the library keeps its own scratch: one
// file-scope device array, FA_NOALLOC_SCRATCH_BYTES long, that exists on every
// GPU that loads this library until the process exits.  The call then runs
// exactly the kernels of fa_bwd with that array as the workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"

namespace fa {
namespace {

// The shared scratch.  On the host this name is only a stand-in for the
// device symbol: host code must pass the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                              float scale, int causal, cudaStream_t stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0)  // invalid sizes: let fa_bwd report which, before any device work
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, nullptr, 0, stream);
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
