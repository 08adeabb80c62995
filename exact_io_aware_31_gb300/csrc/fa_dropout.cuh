// Dropout on the attention probabilities: parameters and the counter-based
// generator of the keep mask.
//
// blog.teqners.com, "The backward pass: recompute instead of read": the
// forward keeps only the dropout generator state and the backward regenerates
// the mask.  The generator is Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), counter-based, so an
// element's bits depend only on (seed, counter).  Element (b, h, query i,
// key j) uses word j mod 4 of the call with counter (j / 4, i, b H + h,
// offset) and key (seed low, seed high); it is kept iff that word is >= thr =
// round(p 2^32), and kept probabilities are scaled by 1 / (1 - p).
#pragma once

#include <cstdint>

namespace fa {

struct DropParams {
  uint32_t thr = 0;      // keep iff word >= thr
  uint32_t k0 = 0;       // seed, low and high 32 bits
  uint32_t k1 = 0;
  uint32_t offset = 0;   // fourth counter word
  float inv_keep = 1.f;  // 1 / (1 - p)
};

#ifdef __CUDACC__
// Philox4x32 round constants from the paper: the two multipliers and the Weyl
// increments of the key.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Ten rounds: (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
// hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)), then the key steps by (W0, W1).
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = c0 * kPhiloxM0, hi0 = __umulhi(c0, kPhiloxM0);
    const uint32_t lo1 = c2 * kPhiloxM1, hi1 = __umulhi(c2, kPhiloxM1);
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return make_uint4(c0, c1, c2, c3);
}
#endif

}  // namespace fa
