// Forward kernel: exact attention with online softmax, tcgen05 + TMA + TMEM.
//
// What it computes follows blog.teqners.com "13% more FLOPs, 5.7x faster ...",
// sections "Softmax is the anti-tiling operation" (running max / normaliser)
// and "FlashAttention's move: rescale the output, too" (rescaled output
// accumulator, division by the normaliser after the last tile), with the loop
// order of lensaml.com "FlashAttention" Step 3 (each CTA owns its Q rows and
// streams K/V tiles past them, writing O once).
//
// Work unit: 256 query rows (two 128-row Q tiles, t = 0, 1) of one (b, h).
// CTA roles (12 warps; warp 11 idle, and warp 10 too at d = 128):
//   warps 0-3  softmax warpgroup for Q tile 0   (thread = one query row)
//   warps 4-7  softmax warpgroup for Q tile 1
//   warp  8    TMA producer: Q tiles, then K_j / V_j into a STAGES-deep ring
//   warp  9    TMEM owner and MMA issuer: every MMA at d = 128; at d = 64
//              the S MMAs (PVW) or every MMA of Q tile 0 (PTI)
//   warp 10    d = 64: the P V MMAs (PVW) or every MMA of Q tile 1 (PTI)
// Tensor memory (512 columns), d = 128: S_t at column 128 t (fp32 scores;
// P_t is written back over its first 64 columns as packed bf16), O_t at
// 256 + 128 t.  Issue order on the tensor pipe alternates the two tiles:
//   S0(j) S1(j) | PV0(j) S0(j+1) | PV1(j) S1(j+1) | PV0(j+1) ...
// so one warpgroup's softmax overlaps the other tile's two MMAs.  Because a
// commit covers every earlier MMA of the issuing thread, the arrival that
// publishes S_t(j+1) also proves PV_t(j) has finished: the softmax warpgroup
// may then rescale O_t in place before it releases P_t(j+1).
// d = 64: S_t at 128 t, P_t at 256 + 64 t, O_t at 384 + 64 t.  With P apart
// from S the order per key tile is S0(j+1) S1(j+1) | PV0(j) | PV1(j): S_t(j+1)
// only waits until the softmax has read S_t(j) into registers, so it runs
// while P_t(j) is computed, and the softmax waits for PV_t(j) (a commit of its
// own) before it rewrites P_t or rescales O_t.  One issuer cannot keep up
// with the softmax warpgroups that share its sub-partition, so d = 64 has
// two.  PVW: the P V MMAs come from a second warp on another sub-partition
// (the S and P V groups need no ordering between them), with K and V
// released separately.  PTI (short causal units, N < 2048): each Q tile has
// an issuer of its own that moves on to the next unit as soon as its tile is
// done, and the longer tile (one key tile more) alternates between the two
// warpgroups from unit to unit, so that neither waits a tile at every unit
// end; K / V slots take one release from each issuer.
// F8 (d = 128): Q and K arrive as E4M3 codes (lensaml.com "FlashAttention",
// "Key ideas", FlashAttention-3's FP8); each tile is one 128-byte-swizzled
// block of 128 one-byte columns, S = Q K^T issues kind::f8f6f4 MMAs (K = 32
// a step), and everything after S is the bf16 path, the two descale factors
// folded into c2 by the host.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_dropout.cuh"
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {

#ifdef FA_TEST_HOOKS
// Test builds only (-DFA_TEST_HOOKS, never the default library): when set,
// softmax warpgroup 0 withholds its first "P ready" arrival of every unit, so
// the MMA warp's bounded wait runs out and the failure-detection path runs.
static __device__ int g_fa_test_withhold_arrival;
#endif

// K / V ring depth at d = 64 (3, 4 and 5 slots measured within 2% of each
// other; 4 leaves room for the TMA-store epilogue's staging boxes).
constexpr int kFwdStagesD64 = 4;

template <int D, bool F8 = false, bool EPI = false>
struct FwdCfg {
  static constexpr int kStages = (D == 128) ? 2 : kFwdStagesD64;
  static constexpr int kQBufs = (D == 128) ? 1 : 2;  // Q buffers per tile (next unit's Q prefetched at d = 64)
  static constexpr int kTileBytes = kTileRows * D * 2;  // a bf16 tile (V; Q and K unless F8)
  static constexpr int kBlocks = D / 64;                // its 128-byte-swizzled 64-column blocks
  // F8: Q and K tiles hold E4M3 codes, one byte an element: 128-column blocks
  static constexpr int kQKBytes = F8 ? kTileRows * D : kTileBytes;
  static constexpr int kQKBlocks = F8 ? D / 128 : kBlocks;
  static constexpr int kQKBlockCols = F8 ? 128 : 64;
  static constexpr int kTmemCols = 512;
  // d = 64: P_t has TMEM columns of its own, so S_t(j+1) is issued as soon as
  // the softmax has read S_t(j) and runs while P_t(j) is being computed.  At
  // d = 128 two S and two O tiles fill the 512 columns and P_t is written over
  // S_t, so S_t(j+1) waits for P_t(j) V_j.
  static constexpr bool kSepP = (D == 64);
  static constexpr int kColS = 0;                   // + 128 t
  static constexpr int kColP = kSepP ? 256 : 0;     // + kPStride t
  static constexpr int kPStride = kSepP ? 64 : 128;
  static constexpr int kColO = kSepP ? 384 : 256;   // + D t
  // 12 warps: two softmax warpgroups and one of producer, MMA issuer(s) and
  // idle warps.  Launched at 168 registers a thread (three warps on each SM
  // sub-partition, one of each warpgroup); the third warpgroup gives
  // registers back so the softmax threads can hold a whole score row (and
  // its exponentials) without spilling: 2 x 128 x kSoftmaxRegs + 128 x
  // kAuxRegs = 384 x 168, which also balances on every sub-partition.
  static constexpr int kThreads = 384;
  static constexpr int kLaunchRegs = 168;
  static constexpr int kAuxRegs = 104;      // the MMA issuer's loop needs about 100
  static constexpr int kSoftmaxRegs = 200;  // no spills at d = 64 or 128 (dropout aside)
  static_assert(2 * 128 * kSoftmaxRegs + 128 * kAuxRegs <= kThreads * kLaunchRegs, "register split");
  // shared memory layout (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQBufs * kQKBytes;
  static constexpr int kOffV = kOffK + kStages * kQKBytes;
  // EPI (d = 64, N < 4096): each softmax warp stages its 32 output rows
  // (bf16, 128-byte swizzled, 4 KiB) and stores them with one TMA copy
  // instead of row-per-thread global stores (32 rows an instruction).  With
  // the short units of those shapes the epilogue is on the critical path
  // once per unit: GPT-2 shape 0.191 -> 0.180 ms; for N >= 4096 it measured
  // up to 2% slower, so those keep the direct stores.
  static constexpr bool kEpiTma = EPI;
  static_assert(!EPI || (D == 64 && !F8), "TMA-store epilogue: d = 64");
  static constexpr int kOffStage = kOffV + kStages * kTileBytes;
  static constexpr int kStageBytes = kEpiTma ? 2 * 4 * 32 * D * 2 : 0;
  static constexpr int kOffBar = kOffStage + kStageBytes;
  static constexpr int kNumBars = 2 * 2 * kQBufs + 4 * kStages + 5 * 2 + 1;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct FwdBars {
  uint64_t* q_full;    // [2][kQBufs]
  uint64_t* q_empty;   // [2][kQBufs]
  uint64_t* k_full;    // [S]
  uint64_t* v_full;    // [S]
  uint64_t* kv_empty;  // [S] K_j read (PTI: one release from each issuer)
  uint64_t* v_empty;   // [S] V_j read (PTI: one release from each issuer)
  uint64_t* s_full;    // [2]
  uint64_t* p_full;    // [2]
  uint64_t* o_full;    // [2]
  uint64_t* s_free;    // [2] (kSepP) the softmax has read S_t
  uint64_t* pv_done;   // [2] (kSepP) P_t V_j has finished
  uint64_t* mma_done;  // [1]
};

// Geometry of one unit.
struct FwdUnit {
  int bh, q0, nq;    // slice, first query row, valid Q tiles (1 or 2)
  int nkv0, nkv1;    // K/V tiles Q tile 0 / 1 visits
  int nkv_max;
  __device__ __forceinline__ int nkv(int t) const { return t ? nkv1 : nkv0; }
};

__device__ __forceinline__ FwdUnit fwd_decode(int pos, int BH, int nqb, int N, int nkv_total, bool causal,
                                              bool block_major) {
  FwdUnit u;
  int r;
  split_unit(pos, BH, nqb, block_major, u.bh, r);
  const int qb = causal ? (nqb - 1 - r) : r;  // heaviest first within a slice when causal
  u.q0 = qb * 2 * kTileRows;
  u.nq = (u.q0 + kTileRows < N) ? 2 : 1;
  int n[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int first = u.q0 + t * kTileRows;
    if (t >= u.nq) {
      n[t] = 0;
    } else if (causal) {
      const int diag = first / kTileRows;
      n[t] = diag + 1 < nkv_total ? diag + 1 : nkv_total;
    } else {
      n[t] = nkv_total;
    }
  }
  u.nkv0 = n[0];
  u.nkv1 = n[1];
  u.nkv_max = n[0] > n[1] ? n[0] : n[1];
  return u;
}

// DROP: dropout on the probabilities (fa_dropout.cuh): the row sum l keeps
// every probability, the P fed to P V keeps only the surviving ones, and the
// epilogue scales O by 1 / (1 - p).
// ISSUE: 0 = one MMA warp, 1 = PVW (a second warp issues every P V),
// 2 = PTI (one issuer per Q tile, d = 64; see the per-tile issuer below).
template <int D, bool CAUSAL, bool DROP, int ISSUE, bool F8 = false, bool EPI = false>
__global__ void __launch_bounds__(FwdCfg<D, F8, EPI>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, int BH, int N, float c2, DropParams dp, int* status) {
  using C = FwdCfg<D, F8, EPI>;
  constexpr bool PVW = ISSUE == 1;
  constexpr bool PTI = ISSUE == 2;
  static_assert((PVW || PTI) == C::kSepP, "d = 64 takes two issuers (P in columns of its own), d = 128 one");
  // A negative scale arrives as a negative c2: the tensor core then computes
  // S negated (Q negated as the A operand) and everything after S uses |c2|,
  // so the row maximum and the masking below are those of a positive scale.
  const uint32_t s_negate = c2 < 0.f ? kIdescNegateA : 0u;
  c2 = fabsf(c2);
  static_assert(!F8 || (D == 128 && !DROP && ISSUE == 0), "FP8 Q, K: d = 128, no dropout, one issuer");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (!smem_base_ok(smem_raw, status)) return;
  uint8_t* sm = smem_raw;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  FwdBars B;
  B.q_full = bars;
  B.q_empty = bars + 2 * C::kQBufs;
  B.k_full = bars + 4 * C::kQBufs;
  B.v_full = B.k_full + C::kStages;
  B.kv_empty = B.v_full + C::kStages;
  B.v_empty = B.kv_empty + C::kStages;
  B.s_full = B.v_empty + C::kStages;
  B.p_full = B.s_full + 2;
  B.o_full = B.p_full + 2;
  B.s_free = B.o_full + 2;
  B.pv_done = B.s_free + 2;
  B.mma_done = B.pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffAbort);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nqb = (N + 2 * kTileRows - 1) / (2 * kTileRows);
  const int nkv_total = (N + kTileRows - 1) / kTileRows;
  const int total_units = BH * nqb;
  const int grid = gridDim.x;
  const bool block_major = block_major_order(CAUSAL, total_units, grid, N);
  // The unit's Q tile that warpgroup / issuer t works on in round `round`:
  // tile t, except with per-tile issuers under the causal mask, where the
  // longer tile (the second one sees one key tile more) alternates between
  // the two from round to round, so that neither runs a tile ahead for good.
  auto slot_of = [](int t, int round) { return (PTI && CAUSAL) ? (t ^ (round & 1)) : t; };

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2 * C::kQBufs; ++q) {
      mbar_init(&B.q_full[q], 1);
      mbar_init(&B.q_empty[q], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&B.s_full[t], 1);
      mbar_init(&B.p_full[t], 128);
      mbar_init(&B.o_full[t], 1);
      mbar_init(&B.s_free[t], 128);
      mbar_init(&B.pv_done[t], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&B.k_full[s], 1);
      mbar_init(&B.v_full[s], 1);
      mbar_init(&B.kv_empty[s], PTI ? 2 : 1);  // PTI: both tiles' issuers release each K / V slot
      mbar_init(&B.v_empty[s], PTI ? 2 : 1);
    }
    mbar_init(B.mma_done, (PVW || PTI) ? 2 : 1);
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
  // Each role's code starts with its warpgroup's register budget: warps 8-11
  // (producer, MMA issuer(s), idle) give registers back, the softmax
  // warpgroups take them.
  if (warp >= 8) {
    regs_dec<C::kAuxRegs>();
    if (warp == 8) {
      // ------------------------------------------------------------ producer --
      if (lane == 0) {
        Tracer tr(3);
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
        uint32_t qcnt[2] = {0, 0};
        uint32_t kv_it = 0;
        bool ok = true;
        for (int round = 0; ok; ++round) {
          const int pos = snake_unit(round, blockIdx.x, grid);
          if (round * grid >= total_units) break;
          if (pos >= total_units) continue;
          const FwdUnit u = fwd_decode(pos, BH, nqb, N, nkv_total, CAUSAL, block_major);
          tr(30);
          #pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int sl = slot_of(t, round);  // the unit's Q tile for warpgroup t's buffers
            if (sl >= u.nq || !ok) continue;
            const int qb = t * C::kQBufs + qcnt[t] % C::kQBufs;
            ok = mbar_wait(&B.q_empty[qb], ((qcnt[t] / C::kQBufs) & 1) ^ 1, status);
            tr(31);
            if (!ok) break;
            uint8_t* dst = sm + C::kOffQ + qb * C::kQKBytes;
            mbar_expect_tx(&B.q_full[qb], C::kQKBytes);
            for (int kb = 0; kb < C::kQKBlocks; ++kb)
              tma_load_3d(dst + kb * kSwzBlockBytes, &tm_q, &B.q_full[qb], kb * C::kQKBlockCols, u.q0 + sl * kTileRows,
                          u.bh);
            ++qcnt[t];
          }
          for (int j = 0; j < u.nkv_max && ok; ++j, ++kv_it) {
            const int st = kv_it % C::kStages;
            const uint32_t ph = (kv_it / C::kStages) & 1;
            tr(32);
            ok = mbar_wait(&B.kv_empty[st], ph ^ 1, status);
            tr(33);
            if (!ok) break;
            uint8_t* kd = sm + C::kOffK + st * C::kQKBytes;
            uint8_t* vd = sm + C::kOffV + st * C::kTileBytes;
            mbar_expect_tx(&B.k_full[st], C::kQKBytes);
            for (int kb = 0; kb < C::kQKBlocks; ++kb)
              tma_load_3d(kd + kb * kSwzBlockBytes, &tm_k, &B.k_full[st], kb * C::kQKBlockCols, j * kTileRows, u.bh);
            if (!(ok = mbar_wait(&B.v_empty[st], ph ^ 1, status))) break;  // K and V slots are released apart
            mbar_expect_tx(&B.v_full[st], C::kTileBytes);
            for (int kb = 0; kb < C::kBlocks; ++kb)
              tma_load_3d(vd + kb * kSwzBlockBytes, &tm_v, &B.v_full[st], kb * 64, j * kTileRows, u.bh);
          }
          if (aborted(abort_flag)) ok = false;
        }
        if (!ok) {
          *abort_flag = 1;
        }
        // Drain: every copy this warp started must have landed before exit.
  #pragma unroll
        for (int t = 0; t < 2; ++t)
          for (uint32_t x = (qcnt[t] > (uint32_t)C::kQBufs ? qcnt[t] - C::kQBufs : 0); x < qcnt[t]; ++x)
            mbar_wait(&B.q_full[t * C::kQBufs + x % C::kQBufs], (x / C::kQBufs) & 1, status);
        for (uint32_t i = (kv_it > (uint32_t)C::kStages ? kv_it - C::kStages : 0); i < kv_it; ++i) {
          mbar_wait(&B.k_full[i % C::kStages], (i / C::kStages) & 1, status);
          mbar_wait(&B.v_full[i % C::kStages], (i / C::kStages) & 1, status);
        }
      }
    } else if (PTI && (warp == 9 || warp == 10)) {
      // ------------------------------------------------ per-tile issuers (PTI) --
      // Warp 9 + w issues every MMA of warpgroup w: S_w(j+1) once the softmax
      // has read S_w(j), P_w V_j once P_w(j) is written, in that order per
      // tile, and moves on to the next unit as soon as its own tile is done.
      // Each K / V slot is released by both issuers (two arrivals): the one
      // whose tile skips key tile j waits until the slot holds it, so that its
      // arrival cannot count towards the slot's previous use.
      const int w = warp - 9;
      const uint32_t idS = idesc_bf16(128, 128, 0, 0) | s_negate;  // S = (+/-) Q K^T, both K-major
      constexpr uint32_t kIdescO = idesc_bf16(128, D, 0, 1);    // O += P V, V is MN-major
      const uint32_t q_s = smem_addr(sm + C::kOffQ);
      const uint32_t k_s = smem_addr(sm + C::kOffK);
      const uint32_t v_s = smem_addr(sm + C::kOffV);
      const uint32_t t_sw = tbase + C::kColS + 128 * w;
      uint32_t qcnt = 0, pcnt = 0, sis = 0, kv_it = 0;
      bool ok = true;
      auto issue_s = [&](int st, int qb) -> bool {  // S_w into its columns, once the softmax read the last one
        if (sis > 0 && !mbar_wait_warp(&B.s_free[w], (sis - 1) & 1, status)) return false;
        tc_fence_after();
        ++sis;
        const uint32_t qa = q_s + qb * C::kQKBytes, ka = k_s + st * C::kQKBytes;
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb)
          mma_ss_run_w<4, 2, 2>(t_sw, sdesc(qa + kb * kSwzBlockBytes, 16, 1024),
                                sdesc(ka + kb * kSwzBlockBytes, 16, 1024), idS, kb > 0);
        mma_commit_w(&B.s_full[w]);
        return true;
      };
      for (int round = 0; ok; ++round) {
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (round * grid >= total_units) break;
        if (pos >= total_units) continue;
        const FwdUnit u = fwd_decode(pos, BH, nqb, N, nkv_total, CAUSAL, block_major);
        const int sl = slot_of(w, round);
        const int n = sl < u.nq ? u.nkv(sl) : 0;  // key tiles this tile visits
        const int qb = w * C::kQBufs + qcnt % C::kQBufs;
        if (n > 0) {
          ok = mbar_wait_warp(&B.q_full[qb], (qcnt / C::kQBufs) & 1, status);
          ++qcnt;
        }
        for (int j = 0; j < u.nkv_max && ok; ++j) {
          const uint32_t it = kv_it + j;
          const int st = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (j >= n) {  // key tile j is the other tile's alone: release this issuer's share of the slot
            ok = mbar_wait_warp(&B.k_full[st], ph, status) && mbar_wait_warp(&B.v_full[st], ph, status);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive(&B.kv_empty[st]);
              mbar_arrive(&B.v_empty[st]);
            }
            __syncwarp();
            continue;
          }
          if (j == 0) {
            ok = mbar_wait_warp(&B.k_full[st], ph, status);
            if (!ok) break;
            tc_fence_after();
            ok = issue_s(st, qb);
            if (!ok) break;
            if (n == 1) mma_commit_w(&B.q_empty[qb]);  // last S of the unit
          }
          if (j + 1 < n) {  // S_w(j+1)
            const uint32_t it1 = it + 1;
            ok = mbar_wait_warp(&B.k_full[it1 % C::kStages], (it1 / C::kStages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            ok = issue_s(it1 % C::kStages, qb);
            if (!ok) break;
            if (j + 2 == n) mma_commit_w(&B.q_empty[qb]);  // last S of the unit
          }
          mma_commit_w(&B.kv_empty[st]);  // K_j: its S was issued before (this commit covers it)
          // P_w V_j
          ok = mbar_wait_warp(&B.p_full[w], pcnt & 1, status);
          ++pcnt;
          if (ok) ok = mbar_wait_warp(&B.v_full[st], ph, status);
          if (!ok) break;
          tc_fence_after();
          mma_ts_run_w<8, 8, 128>(tbase + C::kColO + D * w, tbase + C::kColP + C::kPStride * w,
                                  sdesc(v_s + st * C::kTileBytes, kSwzBlockBytes, 1024), kIdescO, j > 0);
          mma_commit_w(&B.pv_done[w]);
          mma_commit_w(&B.v_empty[st]);
        }
        kv_it += u.nkv_max;
        if (__any_sync(0xffffffffu, aborted(abort_flag))) ok = false;
      }
      if (!ok) *abort_flag = 1;
      mma_commit_w(B.mma_done);
      mbar_wait_warp(B.mma_done, 0, status);
    } else if (!PTI && warp == 9) {
      // ---------------------------------------------------------- MMA issuer --
      {  // whole warp, converged: waits are warp-wide, one elected lane issues
        const uint32_t idS = idesc_bf16(128, 128, 0, 0) | s_negate;  // S = (+/-) Q K^T, both K-major
        constexpr uint32_t kIdescO = idesc_bf16(128, D, 0, 1);    // O += P V, V is MN-major
        const uint32_t q_s = smem_addr(sm + C::kOffQ);
        const uint32_t k_s = smem_addr(sm + C::kOffK);
        const uint32_t v_s = smem_addr(sm + C::kOffV);
        uint32_t qcnt[2] = {0, 0}, pcnt[2] = {0, 0};
        uint32_t sis[2] = {0, 0};  // S_t issued so far (kSepP: each after the softmax read the previous one)
        uint32_t kv_it = 0;
        bool ok = true;
        Tracer tr(2);
        for (int round = 0; ok; ++round) {
          const int pos = snake_unit(round, blockIdx.x, grid);
          if (round * grid >= total_units) break;
          if (pos >= total_units) continue;
          const FwdUnit u = fwd_decode(pos, BH, nqb, N, nkv_total, CAUSAL, block_major);
          tr(10);
          int qbuf[2] = {0, 0};  // Q buffer (t * kQBufs + b) each tile uses in this unit
          #pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= u.nq || !ok) continue;
            qbuf[t] = t * C::kQBufs + qcnt[t] % C::kQBufs;
            ok = mbar_wait_warp(&B.q_full[qbuf[t]], (qcnt[t] / C::kQBufs) & 1, status);
            ++qcnt[t];
          }
          tr(11);
          if (!ok) break;
          auto issue_s = [&](int t, int st) -> bool {
            if (C::kSepP) {  // S_t columns are free once the softmax has read the previous S_t
              if (sis[t] > 0 && !mbar_wait_warp(&B.s_free[t], (sis[t] - 1) & 1, status)) return false;
              tc_fence_after();
            }
            ++sis[t];
            const uint32_t qa = q_s + qbuf[t] * C::kQKBytes, ka = k_s + st * C::kQKBytes;
            // 32 bytes of the 128-byte swizzled rows a step: 16 bf16 or 32 E4M3 elements
            if constexpr (F8) {
  #pragma unroll
              for (int k = 0; k < D / 32; ++k) {
                const uint32_t off = (k / 4) * kSwzBlockBytes + (k % 4) * 32;
                mma_ss_f8_w(tbase + C::kColS + 128 * t, sdesc(qa + off, 16, 1024), sdesc(ka + off, 16, 1024),
                            idesc_e4m3(128, 128), k > 0);
              }
            } else {
              // each 64-column block: four K = 16 steps of 32 bytes inside the swizzle atom
  #pragma unroll
              for (int kb = 0; kb < D / 64; ++kb)
                mma_ss_run_w<4, 2, 2>(tbase + C::kColS + 128 * t, sdesc(qa + kb * kSwzBlockBytes, 16, 1024),
                                    sdesc(ka + kb * kSwzBlockBytes, 16, 1024), idS, kb > 0);
            }
            mma_commit_w(&B.s_full[t]);
            return true;
          };
          // prologue: S_t(0)
          {
            const int st = kv_it % C::kStages;
            ok = mbar_wait_warp(&B.k_full[st], (kv_it / C::kStages) & 1, status);
            if (!ok) break;
            tc_fence_after();
  #pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t < u.nq && ok) ok = issue_s(t, st);
              if (t < u.nq && ok && u.nkv(t) == 1) mma_commit_w(&B.q_empty[qbuf[t]]);  // last S_t of the unit
            }
            if (!ok) break;
            if constexpr (ISSUE == 0) mma_commit_w(&B.kv_empty[st]);  // K_0 read by both S_t(0)
          }
          if constexpr (PVW) {
            // Per key tile j: S_0(j+1), S_1(j+1), each once the softmax has read
            // S_t(j); then K_j is released (its S MMAs were issued before).
            for (int j = 0; j < u.nkv_max && ok; ++j) {
              const uint32_t it = kv_it + j;
              const int st = it % C::kStages;
              const int st_next = (it + 1) % C::kStages;
              bool k_next_ready = false;
  #pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (t >= u.nq || j + 1 >= u.nkv(t) || !ok) continue;
                if (!k_next_ready) {
                  ok = mbar_wait_warp(&B.k_full[st_next], ((it + 1) / C::kStages) & 1, status);
                  if (!ok) break;
                  tc_fence_after();
                  k_next_ready = true;
                }
                tr(40 + t);
                ok = issue_s(t, st_next);
                if (!ok) break;
                if (j + 2 == u.nkv(t)) mma_commit_w(&B.q_empty[qbuf[t]]);  // last S_t of the unit
                tr(24 + t);
              }
              if (ok) mma_commit_w(&B.kv_empty[st]);
            }
          } else
          for (int j = 0; j < u.nkv_max && ok; ++j) {
            const uint32_t it = kv_it + j;
            const int st = it % C::kStages;
            const int st_next = (it + 1) % C::kStages;
            bool v_ready = false, k_next_ready = false;
            #pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= u.nq || !ok) continue;
              if (j >= u.nkv(t)) continue;
              tr(20 + t);
              ok = mbar_wait_warp(&B.p_full[t], pcnt[t] & 1, status);
              tr(22 + t);
              ++pcnt[t];
              if (!ok) break;
              if (!v_ready) {
                ok = mbar_wait_warp(&B.v_full[st], (it / C::kStages) & 1, status);
                if (!ok) break;
                v_ready = true;
              }
              tr(26 + t);
              tc_fence_after();
              // O_t (+)= P_t V_j : A = P_t from TMEM (8 columns per 16 keys), B = V_j MN-major
              const uint32_t va = v_s + st * C::kTileBytes;
              mma_ts_run_w<8, 8, 128>(tbase + C::kColO + D * t, tbase + C::kColS + 128 * t,
                                    sdesc(va, kSwzBlockBytes, 1024), kIdescO, j > 0);
              tr(28 + t);
              if (j + 1 < u.nkv(t)) {
                if (!k_next_ready) {
                  ok = mbar_wait_warp(&B.k_full[st_next], ((it + 1) / C::kStages) & 1, status);
                  if (!ok) break;
                  tc_fence_after();
                  k_next_ready = true;
                }
                tr(40 + t);
                ok = issue_s(t, st_next);
                if (!ok) break;
                if (j + 2 == u.nkv(t)) mma_commit_w(&B.q_empty[qbuf[t]]);  // last S_t of the unit
              } else {
                mma_commit_w(&B.o_full[t]);
              }
              tr(24 + t);
            }
            // V_j is read by both P_t V_j; K_{j+1} by both S_t(j+1), issued
            // here: its slot goes back to the producer a key tile earlier
            // than V_j's, so the copy of K_{j+3} has two key tiles of lead
            // (with one ring of two shared slots the MMA warp waited for
            // K_{j+1} about 1250 cycles a key tile, traced).
            if (ok) {
              mma_commit_w(&B.v_empty[st]);
              if (j + 1 < u.nkv_max) mma_commit_w(&B.kv_empty[st_next]);
            }
          }
          kv_it += u.nkv_max;
          if (__any_sync(0xffffffffu, aborted(abort_flag))) ok = false;
        }
        if (!ok) *abort_flag = 1;
        mma_commit_w(B.mma_done);
        mbar_wait_warp(B.mma_done, 0, status);
      }
    } else if (PVW && warp == 10) {
      // ------------------------------------------------------ P V issuer (PVW) --
      {  // whole warp, converged: waits are warp-wide, one elected lane issues
        constexpr uint32_t kIdescO = idesc_bf16(128, D, 0, 1);  // O += P V, V is MN-major
        const uint32_t v_s = smem_addr(sm + C::kOffV);
        uint32_t pcnt[2] = {0, 0};
        uint32_t kv_it = 0;
        bool ok = true;
        for (int round = 0; ok; ++round) {
          const int pos = snake_unit(round, blockIdx.x, grid);
          if (round * grid >= total_units) break;
          if (pos >= total_units) continue;
          const FwdUnit u = fwd_decode(pos, BH, nqb, N, nkv_total, CAUSAL, block_major);
          for (int j = 0; j < u.nkv_max && ok; ++j) {
            const uint32_t it = kv_it + j;
            const int st = it % C::kStages;
            bool v_ready = false;
  #pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t >= u.nq || j >= u.nkv(t) || !ok) continue;
              ok = mbar_wait_warp(&B.p_full[t], pcnt[t] & 1, status);
              ++pcnt[t];
              if (!ok) break;
              if (!v_ready) {
                ok = mbar_wait_warp(&B.v_full[st], (it / C::kStages) & 1, status);
                if (!ok) break;
                v_ready = true;
              }
              tc_fence_after();
              // O_t (+)= P_t V_j : A = P_t from TMEM (8 columns per 16 keys), B = V_j MN-major
              const uint32_t va = v_s + st * C::kTileBytes;
              mma_ts_run_w<8, 8, 128>(tbase + C::kColO + D * t, tbase + C::kColP + C::kPStride * t,
                                    sdesc(va, kSwzBlockBytes, 1024), kIdescO, j > 0);
              mma_commit_w(&B.pv_done[t]);
            }
            if (ok) mma_commit_w(&B.v_empty[st]);
          }
          kv_it += u.nkv_max;
          if (__any_sync(0xffffffffu, aborted(abort_flag))) ok = false;
        }
        if (!ok) *abort_flag = 1;
        mma_commit_w(B.mma_done);
        mbar_wait_warp(B.mma_done, 0, status);
      }
    }
  } else {
    regs_inc<C::kSoftmaxRegs>();
    // -------------------------------------------------------------- softmax --
    const int t = warp / 4;            // which Q tile this warpgroup owns
    const int quarter = warp % 4;      // TMEM lane quarter
    const int r = quarter * 32 + lane; // row inside the tile
    const uint32_t t_s = tmem_lane_col(tbase, quarter * 32, C::kColS + 128 * t);
    const uint32_t t_o = tmem_lane_col(tbase, quarter * 32, C::kColO + D * t);
    const uint32_t t_p = tmem_lane_col(tbase, quarter * 32, C::kColP + C::kPStride * t);
    uint32_t scnt = 0, ocnt = 0, pvcnt = 0;
    bool ok = true, epi_pending = false;
    Tracer tr(quarter == 0 ? t : -1);
    for (int round = 0; ok; ++round) {
      const int pos = snake_unit(round, blockIdx.x, grid);
      if (round * grid >= total_units) break;
      if (pos >= total_units) continue;
      const FwdUnit u = fwd_decode(pos, BH, nqb, N, nkv_total, CAUSAL, block_major);
      const int sl = slot_of(t, round);  // the unit's Q tile this warpgroup works on
      if (sl >= u.nq) continue;
      const int qi = u.q0 + sl * kTileRows + r;  // this thread's query row
      const int jdiag = (u.q0 + sl * kTileRows) / kTileRows;
      float m_run = -INFINITY;  // running max used by the exponentials (log2 units)
      float l_run = 0.f;        // running normaliser relative to m_run
      for (int j = 0; j < u.nkv(sl); ++j) {
        tr(1);
        ok = mbar_wait_warp(&B.s_full[t], scnt & 1, status);
        tr(2);
        ++scnt;
        if (!ok) break;
        tc_fence_after();
        // Whole S row into registers: four loads in flight, one wait.
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t (&chunk)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]);
          tmem_ld32(t_s + 32 * c, chunk);
        }
        tmem_wait_ld();
        if (C::kSepP) {  // S_t(j) is in registers: the MMA warp may overwrite it with S_t(j+1)
          tc_fence_before();
          mbar_arrive(&B.s_free[t]);
        }
        tr(3);
        float* s = reinterpret_cast<float*>(sv);
        const bool tail = (j == nkv_total - 1) && (N % kTileRows != 0);
        const bool diag = CAUSAL && (j == jdiag);
        if (tail || diag) {
          // Masked keys -> -inf: key kbase + c is visible iff c <= cut.
          const int kbase = j * kTileRows;
          const int lim = CAUSAL ? min(qi, N - 1) : N - 1;
          const int cut = lim - kbase;
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c > cut) ? -INFINITY : s[c];
        }
        // Row max: three-input max, eight independent partial maxima.
        float pm[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pm[e] = max3f(s[2 * e], s[2 * e + 1], -INFINITY);
#pragma unroll
        for (int c = 16; c < 128; c += 2) pm[(c / 2) & 7] = max3f(pm[(c / 2) & 7], s[c], s[c + 1]);
        const float mx = max3f(max3f(pm[0], pm[1], pm[2]), max3f(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        const float mx2 = mx * c2;  // tile max in log2 units (c2 > 0)
        if (C::kSepP && j > 0) {
          // P_t(j - 1) V_{j-1} must be done: it reads the P_t columns about to
          // be rewritten and accumulates into the O_t a rescale would touch.
          ok = mbar_wait_warp(&B.pv_done[t], pvcnt & 1, status);
          ++pvcnt;
          if (!ok) break;
          tc_fence_after();
        }
        if (j == 0) {
          m_run = mx2;
        } else {
          const bool need = mx2 > m_run + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            // O_t is quiescent here (see header): rescale it and l by 2^(m_old - m_new).
            const float m_new = fmaxf(m_run, mx2);
            const float alpha = ex2(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t v[16];
              tmem_ld16(t_o + 16 * c, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float lo, hi;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), a2), lo, hi);
                v[2 * i] = __float_as_uint(lo);
                v[2 * i + 1] = __float_as_uint(hi);
              }
              tmem_st16(t_o + 16 * c, v);
            }
          }
        }
        tr(4);
        // P = 2^(s c2 - m_run) in pairs, summed in fp32, stored as bf16 pairs
        // (over S_t at d = 128) in four 16-column pieces.
        const uint64_t c2x2 = f2_pack(c2, c2);
        const uint64_t negm = f2_pack(-m_run, -m_run);
        uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};  // partial row sums (pairs)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[16];
          uint4 rw = make_uint4(0u, 0u, 0u, 0u);  // DROP: generator words of keys c .. c + 3
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 32 * h + 2 * i;
            const uint64_t x = f2_fma(f2_pack(s[c], s[c + 1]), c2x2, negm);
            float x0, x1;
            f2_unpack(x, x0, x1);
            const uint64_t p = f2_pack(ex2(x0), ex2(x1));
            ls[i & 3] = f2_add(ls[i & 3], p);
            float p0, p1;
            f2_unpack(p, p0, p1);
            if (DROP) {  // one generator call per four keys: words (x, y) for an even pair, (z, w) for an odd one
              if ((i & 1) == 0)
                rw = philox4x32_10((uint32_t)((j * kTileRows + c) >> 2), (uint32_t)qi, (uint32_t)u.bh, dp.offset,
                                   dp.k0, dp.k1);
              if (((i & 1) ? rw.z : rw.x) < dp.thr) p0 = 0.f;
              if (((i & 1) ? rw.w : rw.y) < dp.thr) p1 = 0.f;
            }
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(t_p + 16 * h, pk);
        }
        {
          const uint64_t t01 = f2_add(f2_add(ls[0], ls[1]), f2_add(ls[2], ls[3]));
          float a0, a1;
          f2_unpack(t01, a0, a1);
          l_run += a0 + a1;
        }
        tmem_wait_st();
        tc_fence_before();
#ifdef FA_TEST_HOOKS
        const bool withhold = t == 0 && j == 0 && *reinterpret_cast<volatile int*>(&g_fa_test_withhold_arrival) != 0;
#else
        constexpr bool withhold = false;
#endif
        if (!withhold) mbar_arrive(&B.p_full[t]);
        tr(5);
      }
      if (!ok) break;
      // epilogue: O = O~ / l, lse = (m + log2 l) ln 2
      tr(6);
      if (C::kSepP) {
        ok = mbar_wait_warp(&B.pv_done[t], pvcnt & 1, status);
        ++pvcnt;
      } else {
        ok = mbar_wait_warp(&B.o_full[t], ocnt & 1, status);
        ++ocnt;
      }
      tr(7);
      if (!ok) break;
      tc_fence_after();
      const float inv_l = (DROP ? dp.inv_keep : 1.f) / l_run;
      if constexpr (C::kEpiTma) {
        // This warp's 32 rows into its staging box (16-byte chunk c of row r
        // at chunk c ^ (r % 8): the 128-byte swizzle), then one TMA store of
        // the box; rows past N are clipped by the copy, and a box wholly past
        // the end is not issued.
        uint8_t* stage = sm + C::kOffStage + (t * 4 + quarter) * (32 * D * 2);
        if (lane == 0 && epi_pending) tma_store_wait_read0();  // the previous unit's store has read the box
        __syncwarp();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_o + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int ch = 4 * c + i;  // 16-byte chunk: columns 8 ch .. 8 ch + 7
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * i + 0]) * inv_l, __uint_as_float(v[8 * i + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]) * inv_l, __uint_as_float(v[8 * i + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]) * inv_l, __uint_as_float(v[8 * i + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]) * inv_l, __uint_as_float(v[8 * i + 7]) * inv_l);
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((ch ^ (lane & 7)) << 4)) = w;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int row0 = u.q0 + sl * kTileRows + quarter * 32;
        if (lane == 0 && row0 < N) {
          tma_store_3d(&tm_o, stage, 0, row0, u.bh);
          tma_store_commit();
        }
        epi_pending = true;
      } else {
        __nv_bfloat16* orow = out + ((size_t)u.bh * N + qi) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_o + 32 * c, v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
          if (qi < N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      if (qi < N) lse[(size_t)u.bh * N + qi] = (m_run + __log2f(l_run)) * kLn2;
      tr(8);
      tc_fence_before();
      if (aborted(abort_flag)) ok = false;
    }
    if (!ok) *abort_flag = 1;
    if (C::kEpiTma && lane == 0 && epi_pending) tma_store_wait_all0();  // staged rows read and written
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool DROP, int ISSUE = 0, bool F8 = false, bool EPI = false>
static cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
  using C = FwdCfg<D, F8, EPI>;
  auto kern = fa_fwd_kernel<D, CAUSAL, DROP, ISSUE, F8, EPI>;
  // The register split inside the kernel assumes it was built with exactly
  // kLaunchRegs registers a thread: with fewer, the softmax warpgroups' request
  // for more could never be met.  Refuse to launch such a build.
  static const bool regs_ok = [&] {
    cudaFuncAttributes fa_attr;
    return cudaFuncGetAttributes(&fa_attr, kern) == cudaSuccess && fa_attr.numRegs == C::kLaunchRegs;
  }();
  if (!regs_ok) return cudaErrorInvalidKernelImage;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, C::kThreads, C::kSmemBytes, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o,
                                                       reinterpret_cast<__nv_bfloat16*>(a.o), a.lse, a.BH, a.N,
                                                       a.c2, a.drop, a.status);
  return cudaGetLastError();
}

// d = 64: per-tile issuers for the short causal units (N < 2048: one to
// fifteen key tiles per Q tile), the P V warp otherwise; each measured the
// faster of the two (and of one issuer) on those shapes.  The TMA-store
// epilogue below N = 4096.
template <int D, bool DROP>
static cudaError_t launch_fwd_d(const FwdLaunch& a, cudaStream_t stream) {
  if constexpr (D == 64) {
    if (a.causal && a.N < 2048) return launch_fwd_t<64, true, DROP, 2, false, true>(a, stream);
    if (a.N < 4096)
      return a.causal ? launch_fwd_t<64, true, DROP, 1, false, true>(a, stream)
                      : launch_fwd_t<64, false, DROP, 1, false, true>(a, stream);
    return a.causal ? launch_fwd_t<64, true, DROP, 1>(a, stream) : launch_fwd_t<64, false, DROP, 1>(a, stream);
  } else {
    return a.causal ? launch_fwd_t<D, true, DROP>(a, stream) : launch_fwd_t<D, false, DROP>(a, stream);
  }
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.fp8)  // E4M3 Q and K, d = 128 (checked by the caller)
    return a.causal ? launch_fwd_t<128, true, false, 0, true>(a, stream)
                    : launch_fwd_t<128, false, false, 0, true>(a, stream);
  if (a.dropout) return a.d == 64 ? launch_fwd_d<64, true>(a, stream) : launch_fwd_d<128, true>(a, stream);
  return a.d == 64 ? launch_fwd_d<64, false>(a, stream) : launch_fwd_d<128, false>(a, stream);
}

int fwd_units(int BH, int N) { return BH * ((N + 2 * kTileRows - 1) / (2 * kTileRows)); }

}  // namespace fa

#ifdef FA_TEST_HOOKS
// Test builds only: switch the withheld-arrival hook on (1) or off (0).
extern "C" int fa_test_withhold_arrival(int on) {
  return cudaMemcpyToSymbol(fa::g_fa_test_withhold_arrival, &on, sizeof(int)) == cudaSuccess ? 0 : 4;
}
#endif

#ifdef FA_TRACE
// Trace builds only: phase records of this file's kernels.
extern "C" int fa_trace_dump_fwd(void* host, size_t bytes) { return fa::trace_dump(host, bytes); }
#endif
