// Which CUDA context is current on the calling thread.
//
// Device addresses of the library's file-scope __device__ variables (the
// status word, the scratch array of fa_bwd_noalloc) belong to one context:
// a caller may run the library under a context of its own (driver API), and a
// primary context that is reset and created again gets its variables at new
// addresses.  Host code therefore caches such addresses by the ID the driver
// gives the current context, which is unique for the life of the process.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace fa {

// The current context's unique ID in *id.  If no context is current, the
// current device's primary context is made current first (what the runtime
// does on its first call).  Returns false if the driver cannot say.
inline bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    cudaGetLastError();
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess ||
        get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
      cudaGetLastError();
      return false;
    }
  }
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// A small map from context ID to one device address, filled on first use in
// each context.  Entries are reused round-robin beyond kSlots contexts.
class PerContextAddress {
 public:
  // The address for the current context: the cached one, or `lookup()`'s
  // (a callable returning cudaError_t and writing a void*), cached on success.
  template <class Lookup>
  int get(void** out, Lookup lookup) {
    unsigned long long id = 0;
    if (!current_context_id(&id)) return 1;
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < used_; ++i)
      if (ids_[i] == id) {
        *out = ptrs_[i];
        return 0;
      }
    void* p = nullptr;
    if (lookup(&p) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return 1;
    }
    const int slot = used_ < kSlots ? used_++ : (next_++ % kSlots);
    ids_[slot] = id;
    ptrs_[slot] = p;
    *out = p;
    return 0;
  }

 private:
  static constexpr int kSlots = 64;
  std::mutex mu_;
  unsigned long long ids_[kSlots] = {};
  void* ptrs_[kSlots] = {};
  int used_ = 0;
  int next_ = 0;
};

}  // namespace fa
