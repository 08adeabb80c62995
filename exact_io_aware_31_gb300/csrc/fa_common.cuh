// Shared constants and the persistent schedule of the attention kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#ifdef FA_TRACE
#include <cuda_runtime.h>
#endif

namespace fa {

constexpr int kTileRows = 128;            // rows of every Q / K / V tile (tcgen05 M = 128)
constexpr int kSwzBlockBytes = 128 * 128; // one [128 rows x 64 bf16] 128-byte-swizzled block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Lazy rescaling: the running maximum used for the exponentials is only moved
// when a new row maximum exceeds it by more than this (log2 units), so the
// stored exponentials stay below 2^8 and most tiles skip the O rescale.
constexpr float kRescaleThreshold = 8.0f;

// Static persistent schedule.  Units are numbered head-major (all units of one
// (b, h) slice are consecutive, so their K/V stay hot in L2), heaviest first
// within a slice.  Round r hands units [r*G, (r+1)*G) to the G CTAs, in
// forward order on even rounds and reverse order on odd rounds ("snake"), so a
// CTA that drew a heavy unit in one round draws a light one in the next.
__host__ __device__ inline int snake_unit(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

// Unit order of the persistent schedules.  Slice-major (the units of one
// (b, h) slice next to each other) keeps concurrently running units on the
// same K/V in L2.  Block-major (block k, heaviest first, of every slice, then
// block k + 1) balances the CTAs' totals when the causal mask makes units
// unequal and each CTA runs only a few of them: for B = 1, H = 32, N = 4096
// the busiest CTA's share drops from 1.19x to 1.03x of the mean.  Measured on
// GB300, block-major wins for causal N >= 4096 with few units per CTA (B = 1,
// H = 32, d = 128 forward: 0.130 -> 0.110 ms) and loses at N = 1024, where
// locality matters more (B = 16, H = 16, d = 128: 0.089 -> 0.098 ms).
constexpr int kBlockMajorMinN = 4096;
__host__ __device__ inline bool block_major_order(bool causal, int total_units, int grid, int N) {
  return causal && N >= kBlockMajorMinN && total_units < 16 * grid;
}

// Schedule position -> (slice bh, block index within the slice, 0 = first).
__host__ __device__ inline void split_unit(int pos, int BH, int nblk, bool block_major, int& bh, int& blk) {
  if (block_major) {
    blk = pos / BH;
    bh = pos - blk * BH;
  } else {
    bh = pos / nblk;
    blk = pos - bh * nblk;
  }
}

#ifdef __CUDACC__
// Phase tracing, compiled in only with -DFA_TRACE (a separate build of the
// library, never the default one).  Lane 0 of a traced role appends
// (clock64 << 8 | tag) records for the first kTraceCtas CTAs into this
// translation unit's device buffer, which its fa_trace_dump_<unit>() copies
// out.  Without FA_TRACE a Tracer is an empty object and every call compiles
// away.
constexpr int kTraceCtas = 4;
constexpr int kTraceRoles = 4;
constexpr int kTraceCap = 8192;
#ifdef FA_TRACE
static __device__ unsigned long long g_fa_trace[kTraceCtas * kTraceRoles * kTraceCap];

// Copy (and clear) this translation unit's trace buffer; trace builds only.
static inline int trace_dump(void* host, size_t bytes) {
  const size_t n = sizeof(unsigned long long) * kTraceCtas * kTraceRoles * kTraceCap;
  if (host == nullptr || bytes < n) return 1;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpyFromSymbol(host, g_fa_trace, n) != cudaSuccess) {
    cudaGetLastError();
    return 4;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fa_trace) != cudaSuccess || cudaMemset(p, 0, n) != cudaSuccess) {
    cudaGetLastError();
    return 4;
  }
  return 0;
}
struct Tracer {
  unsigned long long* p;
  int n;
  __device__ explicit Tracer(int role)  // role < 0: not traced
      : p((blockIdx.x < kTraceCtas && role >= 0) ? g_fa_trace + (blockIdx.x * kTraceRoles + role) * kTraceCap
                                                  : nullptr),
        n(0) {}
  __device__ __forceinline__ void operator()(int tag) {
    if (p != nullptr && (threadIdx.x & 31) == 0 && n < kTraceCap)
      p[n++] = (static_cast<unsigned long long>(clock64()) << 8) | static_cast<unsigned>(tag & 0xff);
  }
};
#else
struct Tracer {
  __device__ explicit Tracer(int) {}
  __device__ __forceinline__ void operator()(int) {}
};
#endif

// CTA-local abort flag: set by a role that gave up on a bounded wait, polled
// by the others between units so the whole CTA leaves promptly.
__device__ __forceinline__ bool aborted(const volatile int* flag) { return *flag != 0; }
#endif

}  // namespace fa
