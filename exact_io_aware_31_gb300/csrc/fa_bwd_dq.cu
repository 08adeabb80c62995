// dQ of the deterministic backward: query tiles outer, key tiles inner.
//
// blog.teqners.com, "The backward pass: recompute instead of read": S and P
// are rebuilt tile by tile from Q, K and the saved row statistics.  This
// kernel takes the other loop order from the dK / dV kernel (which holds a
// key tile and streams the query tiles past it): a unit is one 128-row query
// tile of one (b, h), the key tiles stream past it, and dQ accumulates in
// tensor memory in a fixed order, so no reduction between CTAs is needed and
// the result is the same on every run.  Per key tile j:
//     S = Q K_j^T,  dP = dO V_j^T                     (tensor cores, TMEM)
//     dS = 2^(S c2 - lse2) * (dP - D)                  (compute warpgroups)
//     dQ += dS K_j                                     (A = dS from TMEM)
// and at the end of the unit dQ = scale * dQ -> bf16.
//
// Roles (10 warps): two compute warpgroups (thread = query row, warpgroup g
// owning key columns [64 g, 64 g + 64) of S and dP; its dS goes, packed as
// bf16 pairs, over the first half of its own S columns), one TMA producer
// warp (Q, dO and their lse2 / D rows per unit; K, V per key tile through a
// ring), one MMA warp that owns the TMEM: two S banks (key tile j in bank
// j % 2, at columns 0 and 384 at d = 128), dP [128, 256), dQ [256, 256 + d).
// The compute warps release dP as soon as S and dP are in their registers,
// so S and dP of tile j + 1 run on the tensor pipe while dS of tile j is
// computed; dQ += dS_j K_j follows, then S of tile j + 2 over bank j % 2.
// Every MMA here reads one operand from shared memory at up to 128 bytes a
// clock (S and dP both), so keeping the pipe fed, not splitting the MMAs
// (which re-reads Q per part), is what shortens a tile.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {

template <int D>
struct DqCfg {
  static constexpr int kWG = 2;
  static constexpr int kKC = kTileRows / kWG;             // key columns per compute warpgroup
  static constexpr int kComputeWarps = 4 * kWG;
  static constexpr int kComputeThreads = 32 * kComputeWarps;
  static constexpr int kProducerWarp = kComputeWarps;
  static constexpr int kMmaWarp = kComputeWarps + 1;
  static constexpr int kThreads = 32 * (kComputeWarps + 2);
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kBlocks = D / 64;
  static constexpr int kQStages = (D == 64) ? 2 : 1;      // Q / dO / rows of a unit
  // K and V in rings of their own: V_j is last read by dP_j, early, while K_j
  // is read until dQ_j at the end of the tile, and S of tile j + 1 is issued
  // before dQ_j, so the K ring is one deeper to keep its copy ahead.
  static constexpr int kKStages = 3;
  static constexpr int kVStages = (D == 64) ? 3 : 2;
  static constexpr int kTmemCols = 512;
  static constexpr int kColS = 0;                     // S bank 0
  static constexpr int kColDP = 128;
  static constexpr int kColDQ = 256;
  static constexpr int kColS1 = 256 + D;              // S bank 1 (d = 64 leaves 192 columns)
  static constexpr int col_s(int bank) { return bank ? kColS1 : kColS; }
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffK = kOffDO + kQStages * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffRow = kOffV + kVStages * kTileBytes;  // [q stages][-lse2 128 | -D 128] fp32
  static constexpr int kRowBytes = 2 * kTileRows * 4;
  static constexpr int kOffBar = kOffRow + kQStages * kRowBytes;
  static constexpr int kNumBars = 2 * kQStages + 2 * kKStages + 2 * kVStages + 6;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kColS1 + 128 <= kTmemCols, "tensor memory budget");
};

// Unit `pos`: (b, h) slice and query tile; under the causal mask the tiles
// with more visible keys come first within a head (heaviest first).
__device__ __forceinline__ void dq_decode(int pos, int BH, int nqt, bool causal, bool block_major, int& bh, int& i,
                                          int& nkv) {
  int t;
  split_unit(pos, BH, nqt, block_major, bh, t);
  i = causal ? nqt - 1 - t : t;
  nkv = causal ? i + 1 : nqt;
}

// P^T column (bf16 pairs) holding keys 16 k .. 16 k + 15 (each warpgroup
// packs its 64 keys into the first 32 of its own 64 S columns).
__device__ __forceinline__ uint32_t dq_ds_col(int k) { return 64 * (k / 4) + 8 * (k % 4); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(DqCfg<D>::kThreads, 1)
    fa_bwd_dq(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const float* __restrict__ lse2, const float* __restrict__ dsum, __nv_bfloat16* __restrict__ dq, int BH,
              int N, int Npad, float c2, float scale, int* status) {
  using C = DqCfg<D>;
  // A negative scale arrives as a negative c2: S is computed negated (Q
  // negated as the A operand), the exponentials use |c2|, dQ the signed scale.
  const uint32_t s_negate = c2 < 0.f ? kIdescNegateA : 0u;
  c2 = fabsf(c2);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (!smem_base_ok(smem_raw, status)) return;
  uint8_t* sm = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* q_full = bars;                         // [q stages]
  uint64_t* q_empty = q_full + C::kQStages;        // [q stages]
  uint64_t* k_full = q_empty + C::kQStages;        // [K stages]
  uint64_t* k_empty = k_full + C::kKStages;        // [K stages]
  uint64_t* v_full = k_empty + C::kKStages;        // [V stages]
  uint64_t* v_empty = v_full + C::kVStages;        // [V stages]
  uint64_t* s_full = v_empty + C::kVStages;        // S and dP of a key tile in TMEM
  uint64_t* ds_full = s_full + 1;                  // dS of the tile in TMEM (compute threads)
  uint64_t* dq_full = s_full + 2;                  // the unit's dQ complete
  uint64_t* dq_empty = s_full + 3;                 // dQ read out (compute threads)
  uint64_t* mma_done = s_full + 4;
  uint64_t* dp_free = s_full + 5;                  // S and dP of the tile are in registers (compute threads)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffAbort);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nqt = (N + kTileRows - 1) / kTileRows;
  const int total_units = BH * nqt;
  const int grid = gridDim.x;
  // d = 64 backward: slice-major measured faster at N = 4096 (L2 locality)
  const bool block_major = D == 128 && block_major_order(CAUSAL, total_units, grid, N);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(ds_full, C::kComputeThreads);
    mbar_init(dp_free, C::kComputeThreads);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, C::kComputeThreads);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_do);
      uint32_t ucnt = 0, kvit = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        if (round * grid >= total_units) break;
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (pos >= total_units) continue;
        int bh, i, nkv;
        dq_decode(pos, BH, nqt, CAUSAL, block_major, bh, i, nkv);
        const int qs = ucnt % C::kQStages;
        if (!(ok = mbar_wait(&q_empty[qs], ((ucnt / C::kQStages) & 1) ^ 1, status))) break;
        mbar_expect_tx(&q_full[qs], 2 * C::kTileBytes + 2 * kTileRows * 4);
        for (int b = 0; b < C::kBlocks; ++b) {
          tma_load_3d(sm + C::kOffQ + qs * C::kTileBytes + b * kSwzBlockBytes, &tm_q, &q_full[qs], 64 * b,
                      i * kTileRows, bh);
          tma_load_3d(sm + C::kOffDO + qs * C::kTileBytes + b * kSwzBlockBytes, &tm_do, &q_full[qs], 64 * b,
                      i * kTileRows, bh);
        }
        float* rows = reinterpret_cast<float*>(sm + C::kOffRow + qs * C::kRowBytes);
        const size_t roff = (size_t)bh * Npad + (size_t)i * kTileRows;
        bulk_load_1d(rows, lse2 + roff, kTileRows * 4, &q_full[qs]);
        bulk_load_1d(rows + kTileRows, dsum + roff, kTileRows * 4, &q_full[qs]);
        ++ucnt;
        for (int j = 0; j < nkv && ok; ++j, ++kvit) {
          const int ks = kvit % C::kKStages, vs = kvit % C::kVStages;
          if (!(ok = mbar_wait(&k_empty[ks], ((kvit / C::kKStages) & 1) ^ 1, status))) break;
          mbar_expect_tx(&k_full[ks], C::kTileBytes);
          for (int b = 0; b < C::kBlocks; ++b)
            tma_load_3d(sm + C::kOffK + ks * C::kTileBytes + b * kSwzBlockBytes, &tm_k, &k_full[ks], 64 * b,
                        j * kTileRows, bh);
          if (!(ok = mbar_wait(&v_empty[vs], ((kvit / C::kVStages) & 1) ^ 1, status))) break;
          mbar_expect_tx(&v_full[vs], C::kTileBytes);
          for (int b = 0; b < C::kBlocks; ++b)
            tma_load_3d(sm + C::kOffV + vs * C::kTileBytes + b * kSwzBlockBytes, &tm_v, &v_full[vs], 64 * b,
                        j * kTileRows, bh);
        }
        if (aborted(abort_flag)) ok = false;
      }
      if (!ok) *abort_flag = 1;
      // Drain copies in flight (bounded).
      for (uint32_t x = (kvit > (uint32_t)C::kKStages ? kvit - C::kKStages : 0); x < kvit; ++x)
        mbar_wait(&k_full[x % C::kKStages], (x / C::kKStages) & 1, status);
      for (uint32_t x = (kvit > (uint32_t)C::kVStages ? kvit - C::kVStages : 0); x < kvit; ++x)
        mbar_wait(&v_full[x % C::kVStages], (x / C::kVStages) & 1, status);
      for (uint32_t x = (ucnt > (uint32_t)C::kQStages ? ucnt - C::kQStages : 0); x < ucnt; ++x)
        mbar_wait(&q_full[x % C::kQStages], (x / C::kQStages) & 1, status);
    }
  } else if (warp == C::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer --
    {  // whole warp, converged: waits are warp-wide, one elected lane issues
      constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);  // S, dP: A and B K-major over d
      const uint32_t idS = kIdS | s_negate;                   // S = (+/-) Q K^T
      constexpr uint32_t kIdQ = idesc_bf16(128, D, 0, 1);    // dQ += dS K: A from TMEM, B (K) MN-major
      uint32_t ucnt = 0, kvit = 0, dscnt = 0, dqcnt = 0, dpcnt = 0;
      bool ok = true;
      Tracer tr(2);
      for (int round = 0; ok; ++round) {
        if (round * grid >= total_units) break;
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (pos >= total_units) continue;
        int bh, i, nkv;
        dq_decode(pos, BH, nqt, CAUSAL, block_major, bh, i, nkv);
        tr(10);
        const int qs = ucnt % C::kQStages;
        const uint32_t q_s = smem_addr(sm + C::kOffQ + qs * C::kTileBytes);
        const uint32_t do_s = smem_addr(sm + C::kOffDO + qs * C::kTileBytes);
        if (!(ok = mbar_wait_warp(&q_full[qs], (ucnt / C::kQStages) & 1, status))) break;
        // S = Q K^T into S bank it % 2 and dP = dO V^T of key tile `it` (ring
        // slot it % stages).  The bank was last read by dQ of tile it - 2,
        // issued before; dP's columns are rewritten once the compute warps
        // hold the previous tile's dP in registers.
        auto issue_sdp = [&](uint32_t it) -> bool {
          const int ks = it % C::kKStages, vs = it % C::kVStages;
          const uint32_t k_s = smem_addr(sm + C::kOffK + ks * C::kTileBytes);
          const uint32_t v_s = smem_addr(sm + C::kOffV + vs * C::kTileBytes);
          tr(20);
          if (!mbar_wait_warp(&k_full[ks], (it / C::kKStages) & 1, status)) return false;
          tc_fence_after();
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)  // four K = 16 steps of 32 bytes per 64-column block
            mma_ss_run_w<4, 2, 2>(tbase + C::col_s(it & 1), sdesc(q_s + blk * kSwzBlockBytes, 16, 1024),
                                  sdesc(k_s + blk * kSwzBlockBytes, 16, 1024), idS, blk > 0);
          tr(21);
          if (dpcnt > 0 && !mbar_wait_warp(dp_free, (dpcnt - 1) & 1, status)) return false;
          if (!mbar_wait_warp(&v_full[vs], (it / C::kVStages) & 1, status)) return false;
          tc_fence_after();
          tr(22);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            mma_ss_run_w<4, 2, 2>(tbase + C::kColDP, sdesc(do_s + blk * kSwzBlockBytes, 16, 1024),
                                  sdesc(v_s + blk * kSwzBlockBytes, 16, 1024), kIdS, blk > 0);
          ++dpcnt;
          mma_commit_w(s_full);
          mma_commit_w(&v_empty[vs]);  // V of this tile has no later reader
          return true;
        };
        if (!(ok = issue_sdp(kvit))) break;  // the unit's first key tile
        for (int j = 0; j < nkv && ok; ++j, ++kvit) {
          if (j + 1 < nkv && !(ok = issue_sdp(kvit + 1))) break;
          // dQ += dS_j K_j, dS_j packed in TMEM over S bank kvit % 2
          tr(23);
          if (!(ok = mbar_wait_warp(ds_full, dscnt & 1, status))) break;
          tr(24);
          ++dscnt;
          // the first dQ MMA of a unit overwrites the columns: the previous
          // unit's dQ must have been read out
          if (j == 0 && !(ok = mbar_wait_warp(dq_empty, (dqcnt & 1) ^ 1, status))) break;
          tc_fence_after();
          const uint32_t k_s = smem_addr(sm + C::kOffK + (kvit % C::kKStages) * C::kTileBytes);
#pragma unroll
          for (int r = 0; r < 2; ++r)  // runs of four 16-key steps with consecutive dS columns (dq_ds_col)
            mma_ts_run_w<4, 8, 128>(tbase + C::kColDQ, tbase + C::col_s(kvit & 1) + dq_ds_col(4 * r),
                                    sdesc(k_s + r * 4 * 2048, kSwzBlockBytes, 1024), kIdQ, (j > 0 || r > 0));
          mma_commit_w(&k_empty[kvit % C::kKStages]);  // K of this tile has no later reader
        }
        if (!ok) break;
        mma_commit_w(&q_empty[qs]);
        mma_commit_w(dq_full);
        ++dqcnt;
        ++ucnt;
        if (__any_sync(0xffffffffu, aborted(abort_flag))) ok = false;
      }
      if (!ok) *abort_flag = 1;
      mma_commit_w(mma_done);
      mbar_wait_warp(mma_done, 0, status);
    }
  } else {
    // ------------------------------------------------ compute warpgroups --
    const int g = warp / 4;
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;  // query row in the tile
    const uint32_t lanes = (uint32_t)quarter * 32;
    const uint32_t t_dp = tmem_lane_col(tbase, lanes, C::kColDP + C::kKC * g);
    const uint32_t t_dq = tmem_lane_col(tbase, lanes, C::kColDQ + (D / 2) * g);
    uint32_t ucnt = 0, scnt = 0, dqcnt = 0;
    bool ok = true;
    Tracer tr((warp % 4) == 0 ? g : -1);
    for (int round = 0; ok; ++round) {
      if (round * grid >= total_units) break;
      const int pos = snake_unit(round, blockIdx.x, grid);
      if (pos >= total_units) continue;
      int bh, i, nkv;
      dq_decode(pos, BH, nqt, CAUSAL, block_major, bh, i, nkv);
      const int qs = ucnt % C::kQStages;
      const int q = i * kTileRows + r;  // this thread's query
      // -lse2 and -D of this query (copied with the unit's Q / dO)
      const float* rows = reinterpret_cast<const float*>(sm + C::kOffRow + qs * C::kRowBytes);
      float nl2 = 0.f, nd = 0.f;
      const uint64_t c2x2 = f2_pack(c2, c2);
      if (!(ok = mbar_wait_warp(&q_full[qs], (ucnt / C::kQStages) & 1, status))) break;  // the rows are in
      for (int j = 0; j < nkv; ++j) {
        tr(1);
        if (!(ok = mbar_wait_warp(s_full, scnt & 1, status))) break;
        tr(2);
        // this key tile's S bank (tiles alternate between the two)
        const uint32_t t_s = tmem_lane_col(tbase, lanes, C::col_s(scnt & 1) + C::kKC * g);
        ++scnt;
        tc_fence_after();
        if (j == 0) {  // read before the unit's first dS is published (the copy slot is reused after)
          nl2 = rows[r];
          nd = rows[kTileRows + r];
        }
        uint32_t sv[C::kKC], dpv[C::kKC];
#pragma unroll
        for (int c = 0; c < C::kKC / 32; ++c) {
          tmem_ld32(t_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
          tmem_ld32(t_dp + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&dpv[32 * c]));
        }
        tmem_wait_ld();
        // S and dP are in registers: the MMA warp may compute the next dP
        tc_fence_before();
        mbar_arrive(dp_free);
        tr(3);
        const int kbase = j * kTileRows + C::kKC * g;  // first key of this warpgroup's columns
        const bool edge = (CAUSAL && j == i) || (kbase + C::kKC > N);
        const uint64_t nl2x2 = f2_pack(nl2, nl2);
        const uint64_t ndx2 = f2_pack(nd, nd);
        uint32_t pk[C::kKC / 2];
#pragma unroll
        for (int e = 0; e < C::kKC / 2; ++e) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), c2x2, nl2x2), x0,
                    x1);
          float p0 = ex2(x0), p1 = ex2(x1);
          if (edge) {  // masked keys (above the diagonal, or past N) contribute exactly 0
            const int k0 = kbase + 2 * e;
            if (k0 >= N || (CAUSAL && k0 > q)) p0 = 0.f;
            if (k0 + 1 >= N || (CAUSAL && k0 + 1 > q)) p1 = 0.f;
          }
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1),
                           f2_add(f2_pack(__uint_as_float(dpv[2 * e]), __uint_as_float(dpv[2 * e + 1])), ndx2)),
                    d0, d1);
          pk[e] = pack_bf16x2(d0, d1);
        }
        // S of this warpgroup's columns is fully read: dS goes over its first half.
#pragma unroll
        for (int c = 0; c < C::kKC / 32; ++c) tmem_st16(t_s + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * c]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(ds_full);
        tr(5);
      }
      if (!ok) break;
      // ---- epilogue: this warpgroup's half of the dQ columns -> scale * dQ, bf16 ----
      if (!(ok = mbar_wait_warp(dq_full, dqcnt & 1, status))) break;
      ++dqcnt;
      tc_fence_after();
      const bool q_ok = q < N;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(t_dq + 32 * c, v);
        tmem_wait_ld();
        if (c == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(dq_empty);
        }
        if (q_ok) {
          uint4* dst = reinterpret_cast<uint4*>(dq + ((size_t)bh * N + q) * D + (D / 2) * g + 32 * c);
#pragma unroll
          for (int m = 0; m < 4; ++m)
            dst[m] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * m]) * scale, __uint_as_float(v[8 * m + 1]) * scale),
                                pack_bf16x2(__uint_as_float(v[8 * m + 2]) * scale,
                                            __uint_as_float(v[8 * m + 3]) * scale),
                                pack_bf16x2(__uint_as_float(v[8 * m + 4]) * scale,
                                            __uint_as_float(v[8 * m + 5]) * scale),
                                pack_bf16x2(__uint_as_float(v[8 * m + 6]) * scale,
                                            __uint_as_float(v[8 * m + 7]) * scale));
        }
      }
      ++ucnt;
      if (aborted(abort_flag)) ok = false;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

template <int D, bool CAUSAL>
static cudaError_t launch_dq_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = fa_bwd_dq<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<a.dq_grid, C::kThreads, C::kSmemBytes, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, a.lse2, a.dsum,
                                                          reinterpret_cast<__nv_bfloat16*>(a.dq), a.BH, a.N, a.Npad,
                                                          a.c2, a.scale, a.status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_dq_t<64, true>(a, stream) : launch_dq_t<64, false>(a, stream);
  return a.causal ? launch_dq_t<128, true>(a, stream) : launch_dq_t<128, false>(a, stream);
}

int bwd_dq_units(int BH, int N) { return BH * ((N + kTileRows - 1) / kTileRows); }

}  // namespace fa

#ifdef FA_TRACE
// Trace builds only: phase records of this file's kernel.
extern "C" int fa_trace_dump_dq(void* host, size_t bytes) { return fa::trace_dump(host, bytes); }
#endif
