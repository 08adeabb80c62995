// Split-KV forward for decoding: a few new queries against a long key/value
// cache.
//
// lensaml.com "FlashAttention" FAQ "Does FlashAttention help during LLM
// decoding?": each decode step has one query (or a few) per sequence, so the
// score matrix is a row and the cost is reading the cache; Flash-Decoding
// splits that read over many thread blocks.  Here a split is a run of whole
// 128-key tiles of one (b, h); its CTA streams the K/V tiles (TMA, 128-byte
// swizzled boxes, a ring of stages) and keeps the online-softmax state of
// every query of the head (blog.teqners.com, "Softmax is the anti-tiling
// operation" and "FlashAttention's move: rescale the output, too").  With one
// split per head the CTA writes O and lse itself; otherwise each split writes
// its normalised partial output and base-2 logsumexp, and a second kernel
// merges them with the same rescale rule.
//
// At 1-8 queries the work is 4 Nq d FLOPs per key against 4 d bytes of K and
// V, at most 8 FLOP/B: far below the tensor-core ridge, so the contractions
// run on the CUDA cores in fp32 and the kernel is bound by HBM.
//
// fa_decode_split (256 threads, one CTA per (b, h, split)):
//   scores  two threads per key of the tile, each over half of the head
//           dimension (16-byte chunks of the swizzled K row; the queries in
//           shared memory, halves offset by 16 banks), summed with one
//           shuffle; masked keys -inf.
//   softmax per query, across the CTA: tile max, rescale factor, p = 2^(s - m)
//           into shared memory, tile sum.
//   PV      thread = column pair x key group: acc_n += p_n(key) * v(key) over
//           the keys of its group; groups are summed at the end.
// Merging: when a head's splits fit in one thread-block cluster (at most 16
// CTAs that the device can co-schedule), they are launched as one and rank 0
// merges the partials from the other CTAs' shared memory; no workspace, no
// second kernel.  Otherwise each split writes its partial to the workspace and
// fa_decode_combine (one warp per (b, h, query)) merges them; it is launched
// as a programmatic dependent of the split kernel, so its launch overlaps the
// split kernel's tail (it waits for that grid's results first).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {

template <int D>
struct DecCfg {
  static constexpr int kTileKeys = kTileRows;            // 128 keys per tile
  static constexpr int kTileBytes = kTileKeys * D * 2;   // one K or V tile: D / 64 swizzle blocks
  static constexpr int kBlocks = D / 64;
  // K+V stages in flight: 3 x 64 KB at d = 128 (one CTA per SM); 2 x 32 KB at
  // d = 64, small enough for two CTAs per SM (one filling its pipeline while
  // the other streams).
  static constexpr int kStages = (D == 64) ? 2 : 3;
  static constexpr int kCtasPerSm = (D == 64) ? 2 : 1;
  static constexpr int kThreads = 256;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kHalf = D / 2;                    // head dimensions per thread in the score phase
  static constexpr int kQHalfStride = 8 * kHalf + 16;    // floats between the two halves of the queries
  static constexpr int kPairs = D / 2;                   // column pairs (PV phase)
  static constexpr int kGroups = kThreads / kPairs;      // key groups (PV phase): 4 at d = 128, 8 at d = 64
  static constexpr int kOffK = 0;                                  // [stages] K tiles
  static constexpr int kOffV = kOffK + kStages * kTileBytes;       // [stages] V tiles
  static constexpr int kOffQ = kOffV + kStages * kTileBytes;       // [2 halves][8][D / 2] fp32 queries (+pad)
  static constexpr int kOffP = kOffQ + 2 * kQHalfStride * 4;       // [128 keys][8] fp32 probabilities
  static constexpr int kOffRed = kOffP + kTileKeys * 8 * 4;        // [2][warps][8] fp32 reductions
  static constexpr int kOffAcc = kOffRed + 2 * kWarps * 8 * 4;     // [groups][8][D] fp32 partial outputs
  static constexpr int kOffMrg = kOffAcc + kGroups * 8 * D * 4;    // [8][D] partial output + [8] lse2 (cluster merge)
  static constexpr int kOffBar = kOffMrg + (8 * D + 8) * 4;        // [stages] mbarriers
  static constexpr int kOffAbort = kOffBar + 8 * kStages;
  static constexpr int kSmemBytes = kOffAbort + 16;
  static_assert(kSmemBytes * kCtasPerSm <= 232448, "shared memory budget");
  static_assert(kGroups * kPairs == kThreads, "PV mapping");
};

// NQ: queries handled (Nq rounded up to 1, 2, 4 or 8; slots past Nq stay masked).
template <int D, int NQ, bool CAUSAL>
__global__ void __launch_bounds__(256, (D == 64 && NQ <= 4) ? 2 : 1)
    fa_decode_split(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                    float* __restrict__ part_o, float* __restrict__ part_lse2, int BH, int Nq, int Nk, int splits,
                    int cluster_merge, float c2, int* status) {
  using C = DecCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (!smem_base_ok(smem_raw, status)) return;
  uint8_t* sm = smem_raw;
  float* qs = reinterpret_cast<float*>(sm + C::kOffQ);
  float* ps = reinterpret_cast<float*>(sm + C::kOffP);
  float* red = reinterpret_cast<float*>(sm + C::kOffRed);
  float* accs = reinterpret_cast<float*>(sm + C::kOffAcc);
  float* mrg = reinterpret_cast<float*>(sm + C::kOffMrg);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffAbort);

  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int bh = blockIdx.x / splits;
  const int split = blockIdx.x - bh * splits;
  const int tiles = (Nk + kTileRows - 1) / kTileRows;
  const int t0 = (int)((long long)split * tiles / splits);
  const int t1 = (int)((long long)(split + 1) * tiles / splits);
  const int kend = min(t1 * kTileRows, Nk);
  const int shift = Nk - Nq;  // bottom-right causal: key j visible to query n iff j <= n + shift

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Queries -> fp32 in shared memory as [half][query][D / 2] (slots past Nq
  // are zero and stay masked).
  for (int i = tid; i < NQ * D; i += C::kThreads) {
    const int n = i / D, col = i - n * D;
    const int h = col / C::kHalf;
    qs[h * C::kQHalfStride + n * C::kHalf + (col - h * C::kHalf)] =
        (n < Nq) ? __bfloat162float(q[((size_t)bh * Nq + n) * D + col]) : 0.f;
  }
  __syncthreads();
  auto issue = [&](int it) {  // tile it into its stage
    const int st = (it - t0) % C::kStages;
    mbar_expect_tx(&full[st], 2 * C::kTileBytes);
    for (int b = 0; b < C::kBlocks; ++b) {
      tma_load_3d(sm + C::kOffK + st * C::kTileBytes + b * kSwzBlockBytes, &tm_k, &full[st], 64 * b,
                  it * kTileRows, bh);
      tma_load_3d(sm + C::kOffV + st * C::kTileBytes + b * kSwzBlockBytes, &tm_v, &full[st], 64 * b,
                  it * kTileRows, bh);
    }
  };
  if (tid == 0) {
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    for (int it = t0; it < t1 && it < t0 + C::kStages; ++it) issue(it);
  }

  float m_run[NQ], l_run[NQ];  // log2 units; the same in every thread
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    m_run[n] = -INFINITY;
    l_run[n] = 0.f;
  }
  const int cp = tid % C::kPairs;  // PV phase: columns 2 cp, 2 cp + 1
  const int kg = tid / C::kPairs;  // PV phase: keys kg, kg + kGroups, ...
  float acc[NQ][2];
#pragma unroll
  for (int n = 0; n < NQ; ++n) acc[n][0] = acc[n][1] = 0.f;

  int issued = min(t1, t0 + C::kStages);
  for (int it = t0; it < t1; ++it) {
    const int st = (it - t0) % C::kStages;
    if (!mbar_wait(&full[st], ((it - t0) / C::kStages) & 1, status)) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;
    const uint8_t* ks = sm + C::kOffK + st * C::kTileBytes;
    const uint8_t* vs = sm + C::kOffV + st * C::kTileBytes;

    // ---- scores: two threads per key, each over half of the head dimension ----
    // d = 128: half h is swizzle block h, its chunks taken in the order i ^ 4h;
    // d = 64: half h is chunks 4h .. 4h + 3 of the one block.  Either way the
    // eight threads of a quarter-warp hit eight different chunk positions.
    const int kr = tid >> 1, half = tid & 1;
    const int key = it * kTileRows + kr;
    const float* qh = qs + half * C::kQHalfStride;
    float sa[NQ], sb[NQ];  // two partial sums per query (shorter dependency chains)
#pragma unroll
    for (int n = 0; n < NQ; ++n) sa[n] = sb[n] = 0.f;
#pragma unroll
    for (int i = 0; i < C::kHalf / 8; ++i) {
      const int ck = (D == 128) ? (i ^ (4 * half)) : (4 * half + i);  // chunk of the 128-byte row
      const int qc = (D == 128) ? (i ^ (4 * half)) : i;               // chunk within the half
      const uint4 kv = *reinterpret_cast<const uint4*>(ks + ((D == 128) ? half * kSwzBlockBytes : 0) + kr * 128 +
                                                       ((ck ^ (kr & 7)) * 16));
      const __nv_bfloat162* kp = reinterpret_cast<const __nv_bfloat162*>(&kv);
      float kf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(kp[e]);
        kf[2 * e] = f.x;
        kf[2 * e + 1] = f.y;
      }
#pragma unroll
      for (int n = 0; n < NQ; ++n) {
        const float4 qa = *reinterpret_cast<const float4*>(qh + n * C::kHalf + 8 * qc);
        const float4 qb = *reinterpret_cast<const float4*>(qh + n * C::kHalf + 8 * qc + 4);
        float& acc_s = (i & 1) ? sb[n] : sa[n];
        acc_s = fmaf(qa.x, kf[0], acc_s);
        acc_s = fmaf(qa.y, kf[1], acc_s);
        acc_s = fmaf(qa.z, kf[2], acc_s);
        acc_s = fmaf(qa.w, kf[3], acc_s);
        acc_s = fmaf(qb.x, kf[4], acc_s);
        acc_s = fmaf(qb.y, kf[5], acc_s);
        acc_s = fmaf(qb.z, kf[6], acc_s);
        acc_s = fmaf(qb.w, kf[7], acc_s);
      }
    }
    float sc[NQ];
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      const float part = sa[n] + sb[n];
      const float full_dot = part + __shfl_xor_sync(0xffffffffu, part, 1);
      const bool vis = n < Nq && key < kend && (!CAUSAL || key <= n + shift);
      sc[n] = vis ? full_dot * c2 : -INFINITY;
    }
    // ---- tile maximum per query, across the CTA ----
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      float mx = sc[n];
#pragma unroll
      for (int off = 16; off > 0; off /= 2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) red[warp * 8 + n] = mx;
    }
    __syncthreads();
    float m_new[NQ], alpha[NQ];
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      float mt = red[n];
#pragma unroll
      for (int w = 1; w < C::kWarps; ++w) mt = fmaxf(mt, red[w * 8 + n]);
      m_new[n] = fmaxf(m_run[n], mt);
      alpha[n] = (m_run[n] == m_new[n]) ? 1.f : ex2(m_run[n] - m_new[n]);  // 0 when m_run = -inf
      // both threads of a key hold its score; the first one stores and counts it
      const float p = (sc[n] == -INFINITY || half) ? 0.f : ex2(sc[n] - m_new[n]);
      if (!half) ps[kr * 8 + n] = p;
      float sum = p;
#pragma unroll
      for (int off = 16; off > 0; off /= 2) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) red[C::kWarps * 8 + warp * 8 + n] = sum;
    }
    __syncthreads();
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      float lt = 0.f;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) lt += red[C::kWarps * 8 + w * 8 + n];
      l_run[n] = alpha[n] * l_run[n] + lt;
      m_run[n] = m_new[n];
      acc[n][0] *= alpha[n];
      acc[n][1] *= alpha[n];
    }
    // ---- O += P V: thread = column pair cp, keys kg, kg + kGroups, ... ----
    {
      const int cc = (2 * cp) / 8;  // 16-byte chunk of the row holding the pair
      const int within = (2 * cp) % 8;
      const uint8_t* vb = vs + (cc / 8) * kSwzBlockBytes + within * 2;
#pragma unroll 4
      for (int kk = kg; kk < kTileRows; kk += C::kGroups) {
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(vb + kk * 128 + (((cc % 8) ^ (kk & 7)) * 16));
        const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv));
        const float* pk = ps + kk * 8;
        if (NQ >= 4) {
#pragma unroll
          for (int n4 = 0; n4 < NQ; n4 += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pk + n4);
            const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[n4 + e][0] = fmaf(pp[e], vf.x, acc[n4 + e][0]);
              acc[n4 + e][1] = fmaf(pp[e], vf.y, acc[n4 + e][1]);
            }
          }
        } else {
#pragma unroll
          for (int n = 0; n < NQ; ++n) {
            acc[n][0] = fmaf(pk[n], vf.x, acc[n][0]);
            acc[n][1] = fmaf(pk[n], vf.y, acc[n][1]);
          }
        }
      }
    }
    __syncthreads();  // stage st and the probabilities are free again
    if (tid == 0 && issued < t1) issue(issued);
    ++issued;
  }
  if (*abort_flag) {
    // Drain the copies still in flight (bounded) before the CTA exits: the
    // last kStages issued, one per stage, each waited on its latest phase.
    if (tid == 0)
      for (int it = max(t0, min(t1, issued) - C::kStages); it < min(t1, issued); ++it) {
        const int st = (it - t0) % C::kStages;
        mbar_wait(&full[st], ((it - t0) / C::kStages) & 1, status);
      }
    if (cluster_merge) {  // the other CTAs of the cluster wait for this one at both barriers
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  // The merge kernel (a programmatic dependent) may start launching now; it
  // waits for this grid's results before reading them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- sum the key groups, normalise, write ----
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    accs[(kg * 8 + n) * D + 2 * cp] = acc[n][0];
    accs[(kg * 8 + n) * D + 2 * cp + 1] = acc[n][1];
  }
  __syncthreads();
  for (int i = tid; i < Nq * D; i += C::kThreads) {  // i = n * D + column
    const int n = i / D;
    float v = 0.f;
#pragma unroll
    for (int g = 0; g < C::kGroups; ++g) v += accs[g * 8 * D + i];
    float l = 0.f, m = -INFINITY;
#pragma unroll
    for (int nn = 0; nn < NQ; ++nn)
      if (nn == n) {
        l = l_run[nn];
        m = m_run[nn];
      }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    const float lse2 = (l > 0.f) ? m + __log2f(l) : -INFINITY;
    const size_t row = (size_t)bh * Nq + n;
    if (splits == 1) {
      o[row * D + (i - n * D)] = __float2bfloat16_rn(v * inv);
      if (i - n * D == 0) lse[row] = lse2 * kLn2;
    } else if (cluster_merge) {
      mrg[i] = v * inv;
      if (i - n * D == 0) mrg[8 * D + n] = lse2;
    } else {
      const size_t prow = (size_t)split * BH * Nq + row;
      part_o[prow * D + (i - n * D)] = v * inv;
      if (i - n * D == 0) part_lse2[prow] = lse2;
    }
  }
  if (cluster_merge) {
    // The splits of this head form one cluster (rank = split): rank 0 merges
    // the partials straight from the other CTAs' shared memory, with the
    // online-softmax rescale (weights 2^(lse2_r - max)).
    cluster_sync_all();  // every partial is written and visible cluster-wide
    if (cluster_rank() == 0) {
      const uint32_t mrg_addr = smem_addr(mrg);
      for (int i = tid; i < Nq * D; i += C::kThreads) {
        const int n = i / D;
        float m = -INFINITY;
        for (int r = 0; r < splits; ++r) m = fmaxf(m, ld_cluster_f32(mrg_addr + (8 * D + n) * 4, r));
        float l = 0.f, v = 0.f;
        for (int r = 0; r < splits; ++r) {
          const float x = ld_cluster_f32(mrg_addr + (8 * D + n) * 4, r);
          if (x == -INFINITY) continue;
          const float w = ex2(x - m);
          l += w;
          v = fmaf(w, ld_cluster_f32(mrg_addr + i * 4, r), v);
        }
        const size_t row = (size_t)bh * Nq + n;
        o[row * D + (i - n * D)] = __float2bfloat16_rn(v / l);
        if (i - n * D == 0) lse[row] = (m + __log2f(l)) * kLn2;
      }
    }
    cluster_sync_all();  // keep every CTA's shared memory alive until rank 0 has read it
  }
}

// ---------------------------------------------------------------------------
// fa_decode_mma: the split kernel with the two contractions on the tensor
// cores, for 3 to 8 queries.  At eight queries the CUDA-core kernel above is
// bound by its fp32 FMAs (4 Nq d FLOPs a key), not by the cache read.  Here the
// queries sit in the first rows of a 128-row tile whose other rows are zero
// (the copy's out-of-range fill), so S = Q K^T and O += P V are ordinary
// M = 128 tcgen05 MMAs into tensor memory, exactly as in the forward kernel.
// Per 128-key tile the MMAs take about 1000 tensor-core cycles and read
// shared memory about 1200 cycles, below the ~2900 cycles an SM needs to
// stream the tile's 64 KiB of K and V at its share of HBM bandwidth, so the
// kernel stays bound by the cache read.  Rows past Nq are padding: their
// probabilities are written as zero, and rows 32-127, which no warp reads,
// are never stored.
// Roles (4 warps): warp 0 softmax (thread = query row), warp 1 TMA producer
// (the query tile once, then K / V tiles through a ring), warp 2 TMEM owner
// and MMA issuer, warp 3 idle.  Tensor memory: two S banks, [0, 128) and
// [128, 256), tile j in bank j % 2 with P written back over its first 64
// columns as bf16 pairs; O [256, 256 + D).  S of tile j + 1 is issued into
// the other bank as soon as its K has landed, so it runs while the softmax
// computes P of tile j (with one bank, S, softmax and P V of a tile ran one
// after the other: eight queries 36.0 -> 34.7 us a step); S of tile j + 2
// reuses bank j % 2 after P V of tile j in the MMA warp's order.  The
// softmax waits for P V of the previous tile (a commit of its own) before it
// may rescale O in place (lazily, as in the forward).  The splits merge as in the
// CUDA-core kernel: inside a cluster through distributed shared memory (the
// query tile's buffer, free once the last MMA is done, holds each split's
// partial), or through the workspace and the shared merge kernel.
template <int D>
struct DecMmaCfg {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kBlocks = D / 64;
  static constexpr int kStages = 3;
  static constexpr int kThreads = 128;
  static constexpr int kTmemCols = 512;
  static constexpr int kColS = 0;    // + 128 (j % 2): the S bank of tile j
  static constexpr int kColO = 256;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * kStages + 6;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(128, 1)
    fa_decode_mma(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                  float* __restrict__ part_o, float* __restrict__ part_lse2, int BH, int Nq, int Nk, int splits,
                  int cluster_merge, float c2, int* status) {
  using C = DecMmaCfg<D>;
  // A negative scale arrives as a negative c2: S is computed negated on the
  // tensor core and the softmax uses |c2| (its maxima are of the raw scores).
  const uint32_t s_negate = c2 < 0.f ? kIdescNegateA : 0u;
  c2 = fabsf(c2);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (!smem_base_ok(smem_raw, status)) return;
  uint8_t* sm = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;                 // [stages]
  uint64_t* kv_empty = kv_full + C::kStages;    // [stages]
  uint64_t* s_full = kv_empty + C::kStages;  // [2]: one per S bank
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = s_full + 3;
  uint64_t* mma_done = s_full + 4;
  uint64_t* pv_done = s_full + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffAbort);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.x / splits;
  const int split = blockIdx.x - bh * splits;
  const int tiles = (Nk + kTileRows - 1) / kTileRows;
  const int t0 = (int)((long long)split * tiles / splits);
  const int t1 = (int)((long long)(split + 1) * tiles / splits);
  const int nt = t1 - t0;  // >= 1: splits never exceed the tiles
  const int kend = min(t1 * kTileRows, Nk);
  const int shift = Nk - Nq;  // bottom-right causal: key j visible to query n iff j <= n + shift

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(&kv_full[st], 1);
      mbar_init(&kv_empty[st], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 32);
    mbar_init(o_full, 1);
    mbar_init(mma_done, 1);
    mbar_init(pv_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 1) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_expect_tx(q_full, C::kTileBytes);
      for (int b = 0; b < C::kBlocks; ++b)  // rows past Nq arrive zero-filled
        tma_load_3d(sm + C::kOffQ + b * kSwzBlockBytes, &tm_q, q_full, 64 * b, 0, bh);
      bool ok = true;
      int j = 0;
      for (; j < nt && ok; ++j) {
        const int st = j % C::kStages;
        if (!(ok = mbar_wait(&kv_empty[st], ((j / C::kStages) & 1) ^ 1, status))) break;
        if (aborted(abort_flag)) break;
        mbar_expect_tx(&kv_full[st], 2 * C::kTileBytes);
        for (int b = 0; b < C::kBlocks; ++b) {
          tma_load_3d(sm + C::kOffK + st * C::kTileBytes + b * kSwzBlockBytes, &tm_k, &kv_full[st], 64 * b,
                      (t0 + j) * kTileRows, bh);
          tma_load_3d(sm + C::kOffV + st * C::kTileBytes + b * kSwzBlockBytes, &tm_v, &kv_full[st], 64 * b,
                      (t0 + j) * kTileRows, bh);
        }
      }
      if (!ok) *abort_flag = 1;
      // every copy this thread started lands before the CTA exits
      mbar_wait(q_full, 0, status);
      for (int x = (j > C::kStages ? j - C::kStages : 0); x < j; ++x)
        mbar_wait(&kv_full[x % C::kStages], (x / C::kStages) & 1, status);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- MMA issuer --
    const uint32_t idS = idesc_bf16(128, 128, 0, 0) | s_negate;  // S = (+/-) Q K^T, both K-major
    constexpr uint32_t kIdO = idesc_bf16(128, D, 0, 1);            // O += P V, V MN-major
    const uint32_t q_s = smem_addr(sm + C::kOffQ);
    // S of tile j into bank j % 2, once its K / V copy has landed
    auto issue_s = [&](int j) -> bool {
      const int st = j % C::kStages;
      if (!mbar_wait_warp(&kv_full[st], (j / C::kStages) & 1, status)) return false;
      tc_fence_after();
      const uint32_t k_s = smem_addr(sm + C::kOffK + st * C::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)  // four K = 16 steps of 32 bytes per 64-column block
        mma_ss_run_w<4, 2, 2>(tbase + C::kColS + 128 * (j & 1), sdesc(q_s + blk * kSwzBlockBytes, 16, 1024),
                              sdesc(k_s + blk * kSwzBlockBytes, 16, 1024), idS, blk > 0);
      mma_commit_w(&s_full[j & 1]);
      return true;
    };
    bool ok = mbar_wait_warp(q_full, 0, status) && issue_s(0);
    for (int j = 0; j < nt && ok; ++j) {
      const int st = j % C::kStages;
      const uint32_t v_s = smem_addr(sm + C::kOffV + st * C::kTileBytes);
      // S(j + 1) into the other bank: P V(j - 1), its last reader, was issued before
      if (j + 1 < nt && !(ok = issue_s(j + 1))) break;
      if (!(ok = mbar_wait_warp(p_full, j & 1, status))) break;
      tc_fence_after();
      // 16 keys a step: 8 P columns, 16 rows (2048 bytes) of V
      mma_ts_run_w<8, 8, 128>(tbase + C::kColO, tbase + C::kColS + 128 * (j & 1), sdesc(v_s, kSwzBlockBytes, 1024),
                              kIdO, j > 0);
      mma_commit_w(pv_done);
      mma_commit_w(&kv_empty[st]);
      if (__any_sync(0xffffffffu, aborted(abort_flag))) ok = false;
    }
    if (!ok) *abort_flag = 1;
    mma_commit_w(o_full);
    mma_commit_w(mma_done);
    mbar_wait_warp(mma_done, 0, status);
  } else if (warp == 0) {
    // -------------------------------------------------------------- softmax --
    const int n = lane;  // query row
    const uint32_t t_o = tmem_lane_col(tbase, 0, C::kColO);
    float m_run = -INFINITY, l_run = 0.f;  // log2 units
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const uint32_t t_s = tmem_lane_col(tbase, 0, C::kColS + 128 * (j & 1));  // this tile's S bank
      if (!(ok = mbar_wait_warp(&s_full[j & 1], (j >> 1) & 1, status))) break;
      tc_fence_after();
      uint32_t sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(t_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
      tmem_wait_ld();
      float* s = reinterpret_cast<float*>(sv);
      // key kbase + c is visible iff c <= cut (cut < 0: none of the tile)
      const int kbase = (t0 + j) * kTileRows;
      const int lim = (n < Nq) ? (CAUSAL ? min(kend - 1, n + shift) : kend - 1) : -1;
      const int cut = lim - kbase;
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = (c > cut) ? -INFINITY : s[c];
      float pm[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) pm[e] = max3f(s[2 * e], s[2 * e + 1], -INFINITY);
#pragma unroll
      for (int c = 16; c < 128; c += 2) pm[(c / 2) & 7] = max3f(pm[(c / 2) & 7], s[c], s[c + 1]);
      const float mx2 =
          max3f(max3f(pm[0], pm[1], pm[2]), max3f(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7])) * c2;  // -inf if none
      if (j > 0) {  // P V of the previous tile has finished: O is quiescent
        if (!(ok = mbar_wait_warp(pv_done, (j - 1) & 1, status))) break;
        tc_fence_after();
      }
      if (j == 0) {
        m_run = mx2;
      } else {
        const bool need = mx2 > m_run + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_run, mx2);
          const float alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(t_o + 16 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st16(t_o + 16 * c, v);
          }
        }
      }
      // P = 2^(s c2 - m) (0 where masked; a row that has seen no key yet has
      // m = -inf and every entry masked), summed in fp32, stored as bf16 pairs
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      const uint64_t c2x2 = f2_pack(c2, c2), negm = f2_pack(-mref, -mref);
      uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * h + 2 * i;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), c2x2, negm), x0, x1);
          const uint64_t p = f2_pack(ex2(x0), ex2(x1));
          ls[i & 3] = f2_add(ls[i & 3], p);
          float p0, p1;
          f2_unpack(p, p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + 16 * h, pk);
      }
      {
        const uint64_t t01 = f2_add(f2_add(ls[0], ls[1]), f2_add(ls[2], ls[3]));
        float a0, a1;
        f2_unpack(t01, a0, a1);
        l_run += a0 + a1;
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait_warp(o_full, 0, status);
    if (!ok) {
      *abort_flag = 1;
    } else {
      tc_fence_after();
      // this split's output row: normalised O and the base-2 logsumexp
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const float lse2 = (l_run > 0.f) ? m_run + __log2f(l_run) : -INFINITY;
      const size_t row = (size_t)bh * Nq + n;
      const size_t prow = (size_t)split * BH * Nq + row;
      float* mrg = reinterpret_cast<float*>(sm + C::kOffQ);  // [8][D] partial rows + [8] lse2 (cluster merge)
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_o + 32 * c, v);
        tmem_wait_ld();
        if (n < Nq) {
          if (cluster_merge) {
#pragma unroll
            for (int i = 0; i < 32; ++i) mrg[n * D + 32 * c + i] = __uint_as_float(v[i]) * inv;
          } else if (splits == 1) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(o + row * D + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          } else {
            float4* dst = reinterpret_cast<float4*>(part_o + prow * D + 32 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                                   __uint_as_float(v[4 * i + 2]) * inv, __uint_as_float(v[4 * i + 3]) * inv);
          }
        }
      }
      if (n < Nq) {
        if (cluster_merge)
          mrg[8 * D + n] = lse2;
        else if (splits == 1)
          lse[row] = lse2 * kLn2;
        else
          part_lse2[prow] = lse2;
      }
      tc_fence_before();
    }
  }
  if (cluster_merge) {
    // The splits of this head form one cluster (rank = split) and merge their
    // partials through distributed shared memory with the online-softmax
    // rescale (weights 2^(lse2_r - max)).  Every rank writes a slice of the
    // head's output: it first forms the weights of each query from all ranks'
    // lse2, then sums its elements over the ranks.  Every thread of every CTA
    // takes both cluster barriers, also after a timeout (the output is then
    // void and the status word says so).
    cluster_sync_all();
    const uint32_t mrg_addr = smem_addr(sm + C::kOffQ);
    float* wts = reinterpret_cast<float*>(sm + C::kOffK);  // [8][16] weights, [8] 1 / l, [8] m (K ring is free)
    const int t = threadIdx.x;
    if (t < Nq) {
      float m = -INFINITY;
      for (int r = 0; r < splits; ++r) m = fmaxf(m, ld_cluster_f32(mrg_addr + (8 * D + t) * 4, r));
      float l = 0.f;
      for (int r = 0; r < splits; ++r) {
        const float x = ld_cluster_f32(mrg_addr + (8 * D + t) * 4, r);
        const float w = (x == -INFINITY) ? 0.f : ex2(x - m);
        wts[t * 16 + r] = w;
        l += w;
      }
      wts[128 + t] = 1.f / l;
      wts[136 + t] = m;
    }
    __syncthreads();
    const int rank = (int)cluster_rank();
    const int total = Nq * D;
    const int chunk = (total + splits - 1) / splits;
    const int i1 = min(total, (rank + 1) * chunk);
    if (!aborted(abort_flag)) {
      for (int i = rank * chunk + t; i < i1; i += C::kThreads) {
        const int n = i / D;
        float v = 0.f;
        for (int r = 0; r < splits; ++r) v = fmaf(wts[n * 16 + r], ld_cluster_f32(mrg_addr + i * 4, r), v);
        const size_t row = (size_t)bh * Nq + n;
        o[row * D + (i - n * D)] = __float2bfloat16_rn(v * wts[128 + n]);
        if (i - n * D == 0) lse[row] = (wts[136 + n] - __log2f(wts[128 + n])) * kLn2;
      }
    }
    cluster_sync_all();  // keep every CTA's shared memory alive until the others have read it
  }
  // The merge kernel (a programmatic dependent) may start launching; it
  // waits for this grid's results before reading them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

// One warp per (b, h, query): merge the splits' partial outputs.
template <int D>
__global__ void __launch_bounds__(128) fa_decode_combine(const float* __restrict__ part_o,
                                                         const float* __restrict__ part_lse2,
                                                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                         int rows, int splits) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the split kernel's partials are complete
  const int row = blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int s = lane; s < splits; s += 32) m = fmaxf(m, part_lse2[(size_t)s * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float l = 0.f;
  for (int s = lane; s < splits; s += 32) {
    const float x = part_lse2[(size_t)s * rows + row];
    l += (x == -INFINITY) ? 0.f : ex2(x - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off /= 2) l += __shfl_xor_sync(0xffffffffu, l, off);
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float x = part_lse2[(size_t)s * rows + row];
    if (x == -INFINITY) continue;
    const float w = ex2(x - m);
    const float* src = part_o + ((size_t)s * rows + row) * D;
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, src[lane + 32 * e], acc[e]);
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < kPer; ++e) o[(size_t)row * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
  if (lane == 0) lse[row] = (m + __log2f(l)) * kLn2;
}

template <int D, int NQ, bool CAUSAL>
static cudaError_t prepare_split_t(int cluster) {
  using C = DecCfg<D>;
  auto kern = fa_decode_split<D, NQ, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e == cudaSuccess && cluster > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int D, int NQ, bool CAUSAL>
static cudaError_t launch_split_t(const DecLaunch& a, cudaStream_t stream) {
  using C = DecCfg<D>;
  auto kern = fa_decode_split<D, NQ, CAUSAL>;
  cudaError_t e = prepare_split_t<D, NQ, CAUSAL>(a.cluster ? a.splits : 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.BH * a.splits);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of one head form a cluster
  attr[0].val.clusterDim.x = a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, *a.tm_k, *a.tm_v, reinterpret_cast<const __nv_bfloat16*>(a.q),
                            reinterpret_cast<__nv_bfloat16*>(a.o), a.lse, a.part_o, a.part_lse2, a.BH, a.Nq, a.Nk,
                            a.splits, a.cluster, a.c2, a.status);
}

// Clusters of `cluster` split CTAs of this kernel that can be resident at
// once (0: not launchable as a cluster).
template <int D, int NQ, bool CAUSAL>
static int max_clusters_t(int cluster) {
  using C = DecCfg<D>;
  if (prepare_split_t<D, NQ, CAUSAL>(cluster) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fa_decode_split<D, NQ, CAUSAL>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int D, bool CAUSAL>
static int max_clusters_nq(int nq, int cluster) {
  if (nq <= 1) return max_clusters_t<D, 1, CAUSAL>(cluster);
  if (nq <= 2) return max_clusters_t<D, 2, CAUSAL>(cluster);
  if (nq <= 4) return max_clusters_t<D, 4, CAUSAL>(cluster);
  return max_clusters_t<D, 8, CAUSAL>(cluster);
}

template <int D, bool CAUSAL>
static int max_clusters_mma_t(int cluster);

int decode_max_clusters(int d, int nq, int causal, int cluster) {
  if (cluster < 2 || cluster > 16) return 0;
  if (nq >= kDecodeMmaMinNq) {
    if (d == 64) return causal ? max_clusters_mma_t<64, true>(cluster) : max_clusters_mma_t<64, false>(cluster);
    return causal ? max_clusters_mma_t<128, true>(cluster) : max_clusters_mma_t<128, false>(cluster);
  }
  if (d == 64) return causal ? max_clusters_nq<64, true>(nq, cluster) : max_clusters_nq<64, false>(nq, cluster);
  return causal ? max_clusters_nq<128, true>(nq, cluster) : max_clusters_nq<128, false>(nq, cluster);
}

template <int D, bool CAUSAL>
static cudaError_t launch_split_nq(const DecLaunch& a, cudaStream_t stream) {
  if (a.Nq <= 1) return launch_split_t<D, 1, CAUSAL>(a, stream);
  if (a.Nq <= 2) return launch_split_t<D, 2, CAUSAL>(a, stream);
  if (a.Nq <= 4) return launch_split_t<D, 4, CAUSAL>(a, stream);
  return launch_split_t<D, 8, CAUSAL>(a, stream);
}

template <int D, bool CAUSAL>
static cudaError_t prepare_mma_t(int cluster) {
  using C = DecMmaCfg<D>;
  auto kern = fa_decode_mma<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e == cudaSuccess && cluster > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int D, bool CAUSAL>
static cudaError_t launch_mma_t(const DecLaunch& a, cudaStream_t stream) {
  using C = DecMmaCfg<D>;
  cudaError_t e = prepare_mma_t<D, CAUSAL>(a.cluster ? a.splits : 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.BH * a.splits);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of one head form a cluster
  attr[0].val.clusterDim.x = a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fa_decode_mma<D, CAUSAL>, *a.tm_q, *a.tm_k, *a.tm_v,
                            reinterpret_cast<__nv_bfloat16*>(a.o), a.lse, a.part_o, a.part_lse2, a.BH, a.Nq, a.Nk,
                            a.splits, a.cluster, a.c2, a.status);
}

// Clusters of `cluster` tensor-core decode CTAs resident at once (0: none).
template <int D, bool CAUSAL>
static int max_clusters_mma_t(int cluster) {
  using C = DecMmaCfg<D>;
  if (prepare_mma_t<D, CAUSAL>(cluster) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fa_decode_mma<D, CAUSAL>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_decode(const DecLaunch& a, cudaStream_t stream) {
  cudaError_t e;
  if (a.Nq >= kDecodeMmaMinNq) {  // tensor-core contractions (never a cluster)
    if (a.d == 64)
      e = a.causal ? launch_mma_t<64, true>(a, stream) : launch_mma_t<64, false>(a, stream);
    else
      e = a.causal ? launch_mma_t<128, true>(a, stream) : launch_mma_t<128, false>(a, stream);
  } else if (a.d == 64) {
    e = a.causal ? launch_split_nq<64, true>(a, stream) : launch_split_nq<64, false>(a, stream);
  } else {
    e = a.causal ? launch_split_nq<128, true>(a, stream) : launch_split_nq<128, false>(a, stream);
  }
  if (e != cudaSuccess || a.splits == 1 || a.cluster) return e;
  const int rows = a.BH * a.Nq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* po = a.part_o;
  const float* pl = a.part_lse2;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o);
  if (a.d == 64) return cudaLaunchKernelEx(&cfg, fa_decode_combine<64>, po, pl, out, a.lse, rows, a.splits);
  return cudaLaunchKernelEx(&cfg, fa_decode_combine<128>, po, pl, out, a.lse, rows, a.splits);
}

}  // namespace fa
