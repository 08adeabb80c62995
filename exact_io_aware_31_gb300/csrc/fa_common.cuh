// Shared constants and the persistent schedule of the attention kernels.
#pragma once

#include <cstdint>

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

#ifdef __CUDACC__
// CTA-local abort flag: set by a role that gave up on a bounded wait, polled
// by the others between units so the whole CTA leaves promptly.
__device__ __forceinline__ bool aborted(const volatile int* flag) { return *flag != 0; }
#endif

}  // namespace fa
