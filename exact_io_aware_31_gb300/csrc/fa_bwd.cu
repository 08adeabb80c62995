// Backward kernels: gradients of exact attention by recomputation.
//
// blog.teqners.com "13% more FLOPs, 5.7x faster ...", section "The backward
// pass: recompute instead of read": the forward keeps only O and the row
// statistics; the backward rebuilds S and P tile by tile from Q, K, V and
// those statistics (here the logsumexp), trading FLOPs for bytes (lensaml.com
// "FlashAttention" FAQ "Why is FlashAttention faster if it does more FLOPs?").
// The gradient algebra (the pages give none) is the chain rule through
// P = softmax(S), S = scale Q K^T:
//     dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//     dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three launches:
//   1. fa_bwd_pre      D and log2-scaled lse per row (padded to whole tiles),
//                      zero the fp32 dQ accumulator.            (HBM-bound)
//   2. fa_bwd_main     persistent; a unit is one 128-key tile of one (b, h);
//                      K, V stay in shared memory while Q / dO tiles stream
//                      past; dK, dV accumulate in TMEM; dQ partials are added
//                      to the fp32 accumulator with vector reductions.
//   3. fa_bwd_dq_conv  dQ = scale * accumulator -> bf16.       (HBM-bound)
//
// fa_bwd_main roles (10 warps):
//   warps 0-3  compute warpgroup, thread = key row: P^T = 2^(S^T c2 - lse2)
//              -> TMEM (bf16, for dV); dS^T = P^T (dP^T - D) -> shared memory
//              (bf16, 128-byte swizzled, for dK and dQ); dK/dV epilogue
//   warps 4-7  dQ warpgroup, thread = query row: reads each dQ partial from
//              TMEM and reduces it into the accumulator
//   warp  8    TMA producer
//   warp  9    TMEM owner and MMA issuer
// Tensor memory (512 columns): S^T [0,128) with P^T over [0,64); dP^T
// [128,256), reused for the dQ partial once dS^T has left it; dV [256,256+d);
// dK [256+d, 256+2d).  MMA issue order per query tile i:
//   S^T(i) dP^T(i) | dV(i) S^T(i+1) | dK(i) dQ(i) | dP^T(i+1) ...
// so the compute warpgroup's dS(i) overlaps dV(i) and S^T(i+1), and its
// P(i+1) overlaps dK(i), dQ(i) and dP^T(i+1).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {

// ------------------------------------------------------------ preprocess ----
// One warp per group of rows: 8 bf16 (16 bytes) per lane.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const __nv_bfloat16* __restrict__ o,
                                                  const __nv_bfloat16* __restrict__ dout,
                                                  const float* __restrict__ lse, float* __restrict__ lse2,
                                                  float* __restrict__ dsum, float* __restrict__ dq_acc, int BH,
                                                  int N, int Npad) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x % 32;
  const int sub = lane / kLanesPerRow;
  const int part = lane % kLanesPerRow;
  const long long total_rows = (long long)BH * Npad;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long w = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; w * kRowsPerWarp < total_rows;
       w += warps) {
    const long long row = w * kRowsPerWarp + sub;  // index into [BH, Npad]
    const bool in_range = row < total_rows;
    const int bh = in_range ? (int)(row / Npad) : 0;
    const int i = in_range ? (int)(row - (long long)bh * Npad) : 0;
    const bool valid = in_range && i < N;
    float acc = 0.f;
    if (valid) {
      const size_t base = ((size_t)bh * N + i) * D + part * 8;
      const uint4 ov = *reinterpret_cast<const uint4*>(o + base);
      const uint4 dv = *reinterpret_cast<const uint4*>(dout + base);
      const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* dp = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = __bfloat1622float2(op[e]);
        const float2 b = __bfloat1622float2(dp[e]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
      }
      float4* z = reinterpret_cast<float4*>(dq_acc + base);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in_range && part == 0) {
      dsum[row] = valid ? acc : 0.f;
      lse2[row] = valid ? lse[(size_t)bh * N + i] * kLog2e : INFINITY;
    }
  }
}

// ------------------------------------------------------------ dQ convert ----
__global__ void __launch_bounds__(256) fa_bwd_dq_conv(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                      long long n8, float scale) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 r;
    r.x = pack_bf16x2(a.x * scale, a.y * scale);
    r.y = pack_bf16x2(a.z * scale, a.w * scale);
    r.z = pack_bf16x2(b.x * scale, b.y * scale);
    r.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = r;
  }
}

// ------------------------------------------------------------- main kernel --
template <int D>
struct BwdCfg {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kBlocks = D / 64;
  static constexpr int kThreads = 320;
  static constexpr int kTmemCols = 512;
  static constexpr int kColS = 0;
  static constexpr int kColDP = 128;  // also the dQ partial
  static constexpr int kColDV = 256;
  static constexpr int kColDK = 256 + D;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                // [stages]
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;     // [stages]
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;    // 128 x 128 bf16, two swizzle blocks
  static constexpr int kOffBar = kOffDS + 2 * kSwzBlockBytes;
  static constexpr int kNumBars = 2 + 3 * kStages + 11;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;
};

struct BwdUnit {
  int bh, j;      // slice and key tile
  int i0, nq;     // first query tile and number of query tiles
};

__device__ __forceinline__ BwdUnit bwd_decode(int pos, int nkt, bool causal) {
  BwdUnit u;
  u.bh = pos / nkt;
  u.j = pos - u.bh * nkt;  // ascending j = heaviest first under the causal mask
  u.i0 = causal ? u.j : 0;
  u.nq = nkt - u.i0;
  return u;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_main(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const float* __restrict__ lse2, const float* __restrict__ dsum, float* __restrict__ dq_acc,
                __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int BH, int N, int Npad, float c2,
                float scale, int* status) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* do_full = q_full + C::kStages;
  uint64_t* qdo_empty = do_full + C::kStages;
  uint64_t* s_full = qdo_empty + C::kStages;
  uint64_t* p_full = s_full + 1;
  uint64_t* dp_full = s_full + 2;
  uint64_t* ds_full = s_full + 3;
  uint64_t* ds_empty = s_full + 4;
  uint64_t* dq_full = s_full + 5;
  uint64_t* dq_empty = s_full + 6;
  uint64_t* dkdv_full = s_full + 7;
  uint64_t* dkdv_empty = s_full + 8;
  uint64_t* mma_done = s_full + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffAbort);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nkt = (N + kTileRows - 1) / kTileRows;
  const int total_units = BH * nkt;
  const int grid = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&do_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 128);
    mbar_init(ds_empty, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(dkdv_full, 1);
    mbar_init(dkdv_empty, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_do);
      uint32_t ucnt = 0, it = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        if (round * grid >= total_units) break;
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (pos >= total_units) continue;
        const BwdUnit u = bwd_decode(pos, nkt, CAUSAL);
        ok = mbar_wait(kv_empty, (ucnt & 1) ^ 1, status);
        if (!ok) break;
        mbar_expect_tx(kv_full, 2 * C::kTileBytes);
        for (int kb = 0; kb < C::kBlocks; ++kb) {
          tma_load_3d(sm + C::kOffK + kb * kSwzBlockBytes, &tm_k, kv_full, kb * 64, u.j * kTileRows, u.bh);
          tma_load_3d(sm + C::kOffV + kb * kSwzBlockBytes, &tm_v, kv_full, kb * 64, u.j * kTileRows, u.bh);
        }
        ++ucnt;
        for (int x = 0; x < u.nq && ok; ++x, ++it) {
          const int i = u.i0 + x;
          const int st = it % C::kStages;
          ok = mbar_wait(&qdo_empty[st], ((it / C::kStages) & 1) ^ 1, status);
          if (!ok) break;
          mbar_expect_tx(&q_full[st], C::kTileBytes);
          for (int kb = 0; kb < C::kBlocks; ++kb)
            tma_load_3d(sm + C::kOffQ + st * C::kTileBytes + kb * kSwzBlockBytes, &tm_q, &q_full[st], kb * 64,
                        i * kTileRows, u.bh);
          mbar_expect_tx(&do_full[st], C::kTileBytes);
          for (int kb = 0; kb < C::kBlocks; ++kb)
            tma_load_3d(sm + C::kOffDO + st * C::kTileBytes + kb * kSwzBlockBytes, &tm_do, &do_full[st], kb * 64,
                        i * kTileRows, u.bh);
        }
        if (aborted(abort_flag)) ok = false;
      }
      if (!ok) *abort_flag = 1;
      // Drain copies in flight.
      if (ucnt) mbar_wait(kv_full, (ucnt - 1) & 1, status);
      for (uint32_t x = (it > (uint32_t)C::kStages ? it - C::kStages : 0); x < it; ++x) {
        mbar_wait(&q_full[x % C::kStages], (x / C::kStages) & 1, status);
        mbar_wait(&do_full[x % C::kStages], (x / C::kStages) & 1, status);
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T: both K-major over d
      constexpr uint32_t kIdKV = idesc_bf16(128, D, 0, 1);    // dV, dK: B (dO / Q) MN-major
      constexpr uint32_t kIdQ = idesc_bf16(128, D, 1, 1);     // dQ: A (dS) and B (K) MN-major
      const uint32_t k_s = smem_addr(sm + C::kOffK);
      const uint32_t v_s = smem_addr(sm + C::kOffV);
      const uint32_t q_s = smem_addr(sm + C::kOffQ);
      const uint32_t do_s = smem_addr(sm + C::kOffDO);
      const uint32_t ds_s = smem_addr(sm + C::kOffDS);
      uint32_t ucnt = 0, it = 0, pcnt = 0, dscnt = 0, dqcnt = 0;
      bool ok = true;
      auto kmajor = [](uint32_t base, int k) { return base + (k / 4) * kSwzBlockBytes + (k % 4) * 32; };
      auto issue_st = [&](int st) {  // S^T = K Q^T
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tbase + C::kColS, sdesc(kmajor(k_s, k), 16, 1024),
                 sdesc(kmajor(q_s + st * C::kTileBytes, k), 16, 1024), kIdSS, k > 0);
        mma_commit(s_full);
      };
      for (int round = 0; ok; ++round) {
        if (round * grid >= total_units) break;
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (pos >= total_units) continue;
        const BwdUnit u = bwd_decode(pos, nkt, CAUSAL);
        ok = mbar_wait(kv_full, ucnt & 1, status) && mbar_wait(dkdv_empty, (ucnt & 1) ^ 1, status);
        ++ucnt;
        if (!ok) break;
        {
          const int st = it % C::kStages;
          ok = mbar_wait(&q_full[st], (it / C::kStages) & 1, status);
          if (!ok) break;
          tc_fence_after();
          issue_st(st);
        }
        for (int x = 0; x < u.nq && ok; ++x, ++it) {
          const int st = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          // dP^T(i) = V dO^T, into the columns the previous dQ partial used
          ok = mbar_wait(&do_full[st], ph, status) && mbar_wait(dq_empty, (dqcnt & 1) ^ 1, status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tbase + C::kColDP, sdesc(kmajor(v_s, k), 16, 1024),
                   sdesc(kmajor(do_s + st * C::kTileBytes, k), 16, 1024), kIdSS, k > 0);
          mma_commit(dp_full);
          // dV += P^T dO  (A = P^T from TMEM, B = dO MN-major)
          ok = mbar_wait(p_full, pcnt & 1, status);
          ++pcnt;
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTileRows / 16; ++k)
            mma_ts(tbase + C::kColDV, tbase + C::kColS + k * 8,
                   sdesc(do_s + st * C::kTileBytes + k * 2048, kSwzBlockBytes, 1024), kIdKV, (x > 0 || k > 0));
          // S^T(i+1) as early as possible
          if (x + 1 < u.nq) {
            const int st2 = (it + 1) % C::kStages;
            ok = mbar_wait(&q_full[st2], ((it + 1) / C::kStages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            issue_st(st2);
          }
          // dK += dS^T Q ; dQ_part = dS K
          ok = mbar_wait(ds_full, dscnt & 1, status);
          ++dscnt;
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTileRows / 16; ++k)
            mma_ss(tbase + C::kColDK, sdesc(kmajor(ds_s, k), 16, 1024),
                   sdesc(q_s + st * C::kTileBytes + k * 2048, kSwzBlockBytes, 1024), kIdKV, (x > 0 || k > 0));
#pragma unroll
          for (int k = 0; k < kTileRows / 16; ++k)
            mma_ss(tbase + C::kColDP, sdesc(ds_s + k * 2048, kSwzBlockBytes, 1024),
                   sdesc(k_s + k * 2048, kSwzBlockBytes, 1024), kIdQ, k > 0);
          mma_commit(dq_full);
          mma_commit(ds_empty);
          mma_commit(&qdo_empty[st]);
          ++dqcnt;
        }
        if (!ok) break;
        mma_commit(dkdv_full);
        mma_commit(kv_empty);
        if (aborted(abort_flag)) ok = false;
      }
      if (!ok) *abort_flag = 1;
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, status);
    }
  } else if (warp < 4) {
    // ------------------------------------------------- compute warpgroup --
    const int quarter = warp;
    const int r = quarter * 32 + lane;  // key row within the tile
    const uint32_t t_s = tmem_lane_col(tbase, quarter * 32, C::kColS);
    const uint32_t t_dp = tmem_lane_col(tbase, quarter * 32, C::kColDP);
    const uint32_t t_dv = tmem_lane_col(tbase, quarter * 32, C::kColDV);
    const uint32_t t_dk = tmem_lane_col(tbase, quarter * 32, C::kColDK);
    uint8_t* ds_row = sm + C::kOffDS + r * 128;
    const int swz = r & 7;
    uint32_t scnt = 0, dpcnt = 0, dse = 0, ucnt = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      if (round * grid >= total_units) break;
      const int pos = snake_unit(round, blockIdx.x, grid);
      if (pos >= total_units) continue;
      const BwdUnit u = bwd_decode(pos, nkt, CAUSAL);
      const int kr = u.j * kTileRows + r;  // this thread's key
      const bool key_ok = kr < N;
      const float* l2_bh = lse2 + (size_t)u.bh * Npad;
      const float* d_bh = dsum + (size_t)u.bh * Npad;
      for (int x = 0; x < u.nq; ++x) {
        const int i = u.i0 + x;
        const int q0 = i * kTileRows;
        const bool diag = CAUSAL && (i == u.j);
        // ---- P^T = 2^(S^T c2 - lse2), masked entries exactly 0 ----
        ok = mbar_wait_warp(s_full, scnt & 1, status);
        ++scnt;
        if (!ok) break;
        tc_fence_after();
        uint32_t pk[64];  // P^T row, bf16 pairs (also used for dS)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32];
          tmem_ld32(t_s + 32 * c, sv);
          float l2[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 v4 = __ldg(reinterpret_cast<const float4*>(l2_bh + q0 + 32 * c) + e);
            l2[4 * e] = v4.x;
            l2[4 * e + 1] = v4.y;
            l2[4 * e + 2] = v4.z;
            l2[4 * e + 3] = v4.w;
          }
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float p0 = ex2(fmaf(__uint_as_float(sv[2 * e]), c2, -l2[2 * e]));
            float p1 = ex2(fmaf(__uint_as_float(sv[2 * e + 1]), c2, -l2[2 * e + 1]));
            if (diag) {
              const int q = q0 + 32 * c + 2 * e;
              if (q < kr) p0 = 0.f;
              if (q + 1 < kr) p1 = 0.f;
            }
            if (!key_ok) {
              p0 = 0.f;
              p1 = 0.f;
            }
            pk[16 * c + e] = pack_bf16x2(p0, p1);
          }
          uint32_t st16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) st16[e] = pk[16 * c + e];
          tmem_st16(t_s + 16 * c, st16);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
        // ---- dS^T = P^T (dP^T - D) -> shared memory (bf16, swizzled) ----
        ok = mbar_wait_warp(dp_full, dpcnt & 1, status);
        ++dpcnt;
        if (ok) ok = mbar_wait_warp(ds_empty, (dse & 1) ^ 1, status);
        ++dse;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t dpv[32];
          tmem_ld32(t_dp + 32 * c, dpv);
          float dd[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 v4 = __ldg(reinterpret_cast<const float4*>(d_bh + q0 + 32 * c) + e);
            dd[4 * e] = v4.x;
            dd[4 * e + 1] = v4.y;
            dd[4 * e + 2] = v4.z;
            dd[4 * e + 3] = v4.w;
          }
          tmem_wait_ld();
          uint32_t dsk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 pb = *reinterpret_cast<const __nv_bfloat162*>(&pk[16 * c + e]);
            const float2 pf = __bfloat1622float2(pb);
            const float d0 = pf.x * (__uint_as_float(dpv[2 * e]) - dd[2 * e]);
            const float d1 = pf.y * (__uint_as_float(dpv[2 * e + 1]) - dd[2 * e + 1]);
            dsk[e] = pack_bf16x2(d0, d1);
          }
          // queries 32c .. 32c+31 = four 16-byte chunks in swizzle block (32c)/64
          uint8_t* blk = ds_row + ((32 * c) / 64) * kSwzBlockBytes;
          const int ch0 = ((32 * c) % 64) / 8;
#pragma unroll
          for (int m = 0; m < 4; ++m)
            *reinterpret_cast<uint4*>(blk + (((ch0 + m) ^ swz) * 16)) =
                make_uint4(dsk[4 * m], dsk[4 * m + 1], dsk[4 * m + 2], dsk[4 * m + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (!ok) break;
      // ---- epilogue: dV, dK (x scale) -> bf16 ----
      ok = mbar_wait_warp(dkdv_full, ucnt & 1, status);
      ++ucnt;
      if (!ok) break;
      tc_fence_after();
      const size_t rowoff = ((size_t)u.bh * N + kr) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(t_dv + 32 * c, a);
        tmem_ld32(t_dk + 32 * c, b);
        tmem_wait_ld();
        if (key_ok) {
          uint4* dvp = reinterpret_cast<uint4*>(dv + rowoff + 32 * c);
          uint4* dkp = reinterpret_cast<uint4*>(dk + rowoff + 32 * c);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            dvp[m] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * m]), __uint_as_float(a[8 * m + 1])),
                                pack_bf16x2(__uint_as_float(a[8 * m + 2]), __uint_as_float(a[8 * m + 3])),
                                pack_bf16x2(__uint_as_float(a[8 * m + 4]), __uint_as_float(a[8 * m + 5])),
                                pack_bf16x2(__uint_as_float(a[8 * m + 6]), __uint_as_float(a[8 * m + 7])));
            dkp[m] = make_uint4(
                pack_bf16x2(__uint_as_float(b[8 * m]) * scale, __uint_as_float(b[8 * m + 1]) * scale),
                pack_bf16x2(__uint_as_float(b[8 * m + 2]) * scale, __uint_as_float(b[8 * m + 3]) * scale),
                pack_bf16x2(__uint_as_float(b[8 * m + 4]) * scale, __uint_as_float(b[8 * m + 5]) * scale),
                pack_bf16x2(__uint_as_float(b[8 * m + 6]) * scale, __uint_as_float(b[8 * m + 7]) * scale));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(dkdv_empty);
      if (aborted(abort_flag)) ok = false;
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ------------------------------------------------------ dQ warpgroup --
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;  // query row within the tile
    const uint32_t t_dq = tmem_lane_col(tbase, quarter * 32, C::kColDP);
    uint32_t qcnt = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      if (round * grid >= total_units) break;
      const int pos = snake_unit(round, blockIdx.x, grid);
      if (pos >= total_units) continue;
      const BwdUnit u = bwd_decode(pos, nkt, CAUSAL);
      for (int x = 0; x < u.nq; ++x) {
        const int q = (u.i0 + x) * kTileRows + r;
        ok = mbar_wait_warp(dq_full, qcnt & 1, status);
        ++qcnt;
        if (!ok) break;
        tc_fence_after();
        float* dst = dq_acc + ((size_t)u.bh * N + q) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_dq + 32 * c, v);
          tmem_wait_ld();
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(dq_empty);
          }
          if (q < N) {
#pragma unroll
            for (int m = 0; m < 8; ++m)
              red_add_v4(dst + 32 * c + 4 * m, __uint_as_float(v[4 * m]), __uint_as_float(v[4 * m + 1]),
                         __uint_as_float(v[4 * m + 2]), __uint_as_float(v[4 * m + 3]));
          }
        }
      }
      if (aborted(abort_flag)) ok = false;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

template <int D, bool CAUSAL>
static cudaError_t launch_main_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = fa_bwd_main<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, C::kThreads, C::kSmemBytes, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, a.lse2, a.dsum,
                                                       a.dq_acc, reinterpret_cast<__nv_bfloat16*>(a.dk),
                                                       reinterpret_cast<__nv_bfloat16*>(a.dv), a.BH, a.N, a.Npad,
                                                       a.c2, a.scale, a.status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t stream) {
  auto o = reinterpret_cast<const __nv_bfloat16*>(a.o);
  auto dout = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  if (a.d == 64)
    fa_bwd_pre<64><<<a.pre_grid, 256, 0, stream>>>(o, dout, a.lse, a.lse2, a.dsum, a.dq_acc, a.BH, a.N, a.Npad);
  else
    fa_bwd_pre<128><<<a.pre_grid, 256, 0, stream>>>(o, dout, a.lse, a.lse2, a.dsum, a.dq_acc, a.BH, a.N, a.Npad);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdLaunch& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_main_t<64, true>(a, stream) : launch_main_t<64, false>(a, stream);
  return a.causal ? launch_main_t<128, true>(a, stream) : launch_main_t<128, false>(a, stream);
}

cudaError_t launch_bwd_conv(const BwdLaunch& a, cudaStream_t stream) {
  const long long n8 = (long long)a.BH * a.N * a.d / 8;
  fa_bwd_dq_conv<<<a.pre_grid, 256, 0, stream>>>(a.dq_acc, reinterpret_cast<__nv_bfloat16*>(a.dq), n8, a.scale);
  return cudaGetLastError();
}

int bwd_units(int BH, int N) { return BH * ((N + kTileRows - 1) / kTileRows); }

}  // namespace fa
