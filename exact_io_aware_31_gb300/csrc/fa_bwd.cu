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
//   1. fa_bwd_pre      -D and -lse*log2(e) per row (padded to whole tiles with
//                      0 and -inf), zero the fp32 dQ accumulator. (HBM-bound)
//   2. fa_bwd_main     persistent; a unit is one 128-key tile of one (b, h);
//                      K, V stay in shared memory while Q / dO tiles stream
//                      past; dK, dV accumulate in TMEM; each query tile's dQ
//                      partial is added to the fp32 accumulator.
//   3. fa_bwd_dq_conv  dQ = scale * accumulator -> bf16.       (HBM-bound)
//
// fa_bwd_main roles (n compute warpgroups: 2 at d = 64, 4 at d = 128):
//   warps 0 .. 4n-1   compute warpgroups, thread = key row, warpgroup g owning
//                     query columns [g 128/n, (g+1) 128/n):
//                     P^T = 2^(S^T c2 - lse2) -> TMEM (bf16, over the first
//                     half of its own S^T columns, for dV);
//                     dS^T = P^T (dP^T - D) -> shared memory (bf16, 128-byte
//                     swizzled, for dK and dQ); at d = 128 they also drain
//                     their columns of the previous tile's dQ^T partial with
//                     coalesced reductions; their share of the dK/dV epilogue
//   warp  4n          TMA producer (K/V per unit, double-buffered at d = 64;
//                     Q, dO and their lse2 / D rows per query tile)
//   warp  4n+1        TMEM owner and MMA issuer
//   warps 4n+2 ..     (d = 64) dQ warpgroup, thread = query row: reads each dQ
//                     partial, releases it, stages it in shared memory and
//                     adds it with a tensor reduce-add
// Tensor memory (512 columns): S^T [0,128); dP^T [128,256); dV [256,256+d);
// dK [256+d, 256+2d); the dQ partial in [384,448) at d = 64, and over dP^T at
// d = 128 (no columns left).
// MMA issue order per query tile i:
//   d = 64:  dV(i) S^T(i+1) | dK(i) dP^T(i+1) dQ(i) | dV(i+1) ...
//            (dP^T(i+1) as soon as dS(i) is in shared memory; dS is
//            double-buffered, so dS(i+1) does not wait for dK(i), dQ(i))
//   d = 128: dP^T(i) | dV(i) S^T(i+1) | dK(i) dQ^T(i) | dP^T(i+1) ...
//            (dP^T(i+1) waits until dQ^T(i), in its columns, is drained)
// Q(i) and dO(i) are released right after dK(i), their last reader.
// so the compute warpgroups' dS(i) overlaps dV(i) and S^T(i+1), and their
// P(i+1) overlaps the MMAs that follow dS(i).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_dropout.cuh"
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {

// Compute warpgroups of the main kernel at d = 64 and d = 128; warpgroup g
// owns query columns [g 128/n, (g+1) 128/n) of every tile.  More warpgroups
// hide more of the TMEM-load, MUFU and shared-memory latency of the P and dS
// phases, at fewer registers per thread.
constexpr int kBwdComputeWgD64 = 2;
constexpr int kBwdComputeWgD128 = 4;
// d = 128: of a thread's dQ^T reductions of the previous query tile, this
// many go out at once after the partial is read from TMEM; the rest are
// spread evenly over the chunks of the next dS loop (fewer values stay live
// through it, and the reductions overlap its arithmetic).
constexpr int kBwdDqImmediate = 16;

// ------------------------------------------------------------ preprocess ----
// One warp per group of rows: 8 bf16 (16 bytes) per lane.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const __nv_bfloat16* __restrict__ o,
                                                  const __nv_bfloat16* __restrict__ dout,
                                                  const float* __restrict__ lse, float* __restrict__ lse2,
                                                  float* __restrict__ dsum, float* __restrict__ dq_acc, int BH,
                                                  int N, int Npad, int zero_dq) {
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
      if (zero_dq) {
        float4* z = reinterpret_cast<float4*>(dq_acc + base);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in_range && part == 0) {
      dsum[row] = valid ? -acc : 0.f;
      lse2[row] = valid ? -lse[(size_t)bh * N + i] * kLog2e : -INFINITY;
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
// DQ = false builds the dK / dV-only variant of the deterministic backward
// (dQ then comes from fa_bwd_dq, with no reductions at all).
template <int D, bool DQ = true>
struct BwdCfg {
  static constexpr int kStages = 2;                   // Q / dO (+ lse2 / D rows) ring
  static constexpr int kKvStages = (D == 64) ? 2 : 1; // K / V buffers (next unit prefetch)
  static constexpr bool kDqAliasesDp = DQ && (D == 128);  // no spare TMEM columns at d = 128
  // At d = 128 the partial is computed transposed, dQ^T = K^T dS^T (TMEM lanes =
  // head dimension), so a warp's reductions cover contiguous 128-byte rows of
  // the accumulator; at d = 64 (M = 64 is not used) it is dQ = dS K, staged in
  // shared memory and added with a tensor reduce-add.
  static constexpr bool kDqTransposed = (D == 128);
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kBlocks = D / 64;
  // d = 64: a dedicated dQ warpgroup (the last four warps) drains each partial
  // through the staging buffers with tensor reduce-adds (asynchronous, so it
  // never waits on them); d = 128: the compute warpgroups drain it with
  // coalesced reductions (a dedicated warpgroup measured slower there).
  static constexpr bool kDqWarpgroup = DQ && !kDqTransposed;
  // With the dQ warpgroup, that warpgroup also writes each unit's dK and dV
  // (through its staging buffer, after the unit's last dQ partial), so the
  // compute warpgroups go straight on to the next unit: at the unit ends of
  // the causal GPT-2 shape the compute warps' own epilogue took about a
  // sixth of their time.
  static constexpr bool kEpiDqWg = kDqWarpgroup;
  // d = 64: dK / dV leave through the dS buffer (free once the unit's last
  // MMAs are done) as two 64-column boxes with TMA stores; at d = 128 they
  // do not fit there and each thread stores its own row.
  static constexpr bool kEpiTma = (D == 64);
  static constexpr int kWG = (D == 64) ? kBwdComputeWgD64 : kBwdComputeWgD128;  // compute warpgroups
  static_assert(kWG == 2 || kWG == 4, "2 or 4 compute warpgroups");
  static constexpr int kQCols = kTileRows / kWG;  // query columns per compute warpgroup
  static constexpr int kDCols = D / kWG;          // dV / dK columns per compute warpgroup (epilogue)
  static constexpr int kComputeWarps = 4 * kWG;
  static constexpr int kComputeThreads = 32 * kComputeWarps;
  static constexpr int kProducerWarp = kComputeWarps;
  static constexpr int kMmaWarp = kComputeWarps + 1;
  static constexpr int kDqWarp0 = kComputeWarps + 2;  // first warp of the dQ warpgroup
  // d = 128 with dQ: 20 warps (four compute warpgroups and one of producer,
  // MMA issuer and two idle warps), launched at 96 registers a thread (five
  // warps on each SM sub-partition, one of each warpgroup); the last
  // warpgroup gives registers back (64) and the compute warps take them
  // (104): their held dQ values and dS loop otherwise spill into local
  // memory, through the same LSU path the dQ reductions take.
  // 4 x 128 x 104 + 128 x 64 = 640 x 96, on the block and on every
  // sub-partition.  (Without dQ the 96 registers suffice.)
  static constexpr bool kRegSplit = (D == 128) && DQ;
  static constexpr int kThreads = kRegSplit ? 640 : 32 * (kComputeWarps + 2 + (kDqWarpgroup ? 4 : 0));
  static constexpr int kLaunchRegs = 96;
  static constexpr int kAuxRegs = 64;
  static constexpr int kComputeRegs = 104;
  static_assert(!kRegSplit || 4 * 128 * kComputeRegs + 128 * kAuxRegs <= kThreads * kLaunchRegs, "register split");
  static constexpr int kTmemCols = 512;
  static constexpr int kColS = 0;     // S^T; P^T of warpgroup g over columns [kQCols g, kQCols g + kQCols / 2)
  static constexpr int kColDP = 128;  // dP^T
  static constexpr int kColDV = 256;
  static constexpr int kColDK = 256 + D;
  static constexpr int kColDQ = !DQ ? 0 : kDqAliasesDp ? kColDP : 256 + 2 * D;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKvStages * kTileBytes;
  static constexpr int kOffQ = kOffV + kKvStages * kTileBytes;    // [stages]
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;     // [stages]
  // d = 64: dP^T(i+1) is issued as soon as dS(i) is in shared memory (ahead
  // of dK(i), dQ(i)), and dS is double-buffered so dS(i+1) need not wait for
  // those two to finish reading dS(i).  At d = 128 the dQ^T partial occupies
  // the dP^T columns, so dP^T(i+1) waits until dQ^T(i) has been drained.
  static constexpr bool kEarlyDp = !kDqAliasesDp;
  // dS is packed as bf16 pairs into the first half of each warpgroup's own
  // dP^T columns (read into registers just before) and dK takes its A operand
  // from tensor memory, so shared memory does not carry the dK MMA's A reads
  // (32 KiB a tile pair, in kernels whose MMAs otherwise read shared memory
  // at its full rate).  dP^T(i+1) overwrites those columns after dK(i) in
  // issue order.  With dQ, dS also goes to shared memory: dQ needs it as a B
  // operand, which only shared memory can hold.  (Without dQ, the dK / dV
  // kernel of the deterministic backward, shared memory carries no dS at
  // all.)  The fused d = 128 kernel keeps dK's A in shared memory: there the
  // tensor-memory copy measured no faster.
  static constexpr bool kDsTmem = !DQ || D == 64;
  static constexpr bool kDsSmem = DQ;
  static constexpr int kDsBufs = (kEarlyDp && D == 64) ? 2 : 1;  // no room for a second one at d = 128
  static constexpr int kDsBytes = 2 * kSwzBlockBytes;              // 128 x 128 bf16 dS^T, two swizzle blocks
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;    // [kDsBufs]
  // d = 64: staging buffer of the dQ partial (128 rows x 64 fp32, as two
  // 128-byte-swizzled 32-column boxes) for the tensor reduce-add.
  static constexpr int kDqStageBytes = (DQ && !kDqTransposed) ? kTileRows * D * 4 : 0;
  static constexpr int kOffDQS = kOffDS + kDsBufs * kDsBytes;
  static constexpr int kOffRow = kOffDQS + kDqStageBytes;        // [stages][lse2 128 | D 128] fp32
  static constexpr int kRowBytes = 2 * kTileRows * 4;
  static constexpr int kOffBar = kOffRow + kStages * kRowBytes;
  static constexpr int kNumBars = 2 * kKvStages + 3 * kStages + 16;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(!DQ || kColDQ + D <= kTmemCols, "tensor memory budget");
};

struct BwdUnit {
  int bh, j;      // slice and key tile
  int i0, nq;     // first query tile and number of query tiles
  int rot;        // the unit visits its query tiles starting at i0 + rot, wrapping
  // x-th query tile the unit visits.  Without the causal mask every key tile
  // of a slice visits all query tiles; starting unit j at tile j keeps the
  // units that run at the same time off the same dQ rows (reductions to one
  // L2 line serialise).  Under the mask unit j already starts at its own
  // diagonal tile j.
  __device__ __forceinline__ int qtile(int x) const {
    const int k = x + rot;
    return i0 + (k >= nq ? k - nq : k);
  }
};

__device__ __forceinline__ BwdUnit bwd_decode(int pos, int BH, int nkt, bool causal, bool block_major) {
  BwdUnit u;
  split_unit(pos, BH, nkt, block_major, u.bh, u.j);  // ascending j = heaviest first under the causal mask
  u.i0 = causal ? u.j : 0;
  u.nq = nkt - u.i0;
  u.rot = causal ? 0 : u.j;
  return u;
}

// P^T column (32-bit, bf16 pairs) holding queries 16 k .. 16 k + 15: the
// warpgroup owning them (QC query columns each) packs its P^T into the first
// half of its own S^T columns.
template <int QC>
__device__ __forceinline__ uint32_t pt_col(int k) {
  return QC * (k / (QC / 16)) + 8 * (k % (QC / 16));
}

// DROP: gradients of the forward with dropout (fa_dropout.cuh): dV takes
// P o M / (1 - p), and dS = P o (dP o M / (1 - p) - D).
template <int D, bool CAUSAL, bool DQ, bool DROP>
__global__ void __launch_bounds__(BwdCfg<D, DQ>::kThreads, 1)
    fa_bwd_main(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dqacc, const __grid_constant__ CUtensorMap tm_dk,
                const __grid_constant__ CUtensorMap tm_dv, const float* __restrict__ lse2,
                const float* __restrict__ dsum, float* __restrict__ dq_acc,
                __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int BH, int N, int Npad, float c2,
                float scale, DropParams dp, int* status) {
  using C = BwdCfg<D, DQ>;
  // A negative scale arrives as a negative c2: S^T is computed negated (K
  // negated as the A operand) and P uses |c2|; dK and dQ take the signed scale.
  const uint32_t s_negate = c2 < 0.f ? kIdescNegateA : 0u;
  c2 = fabsf(c2);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (!smem_base_ok(smem_raw, status)) return;
  uint8_t* sm = smem_raw;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* kv_full = bars;                       // [kv stages]
  uint64_t* kv_empty = kv_full + C::kKvStages;    // [kv stages]
  uint64_t* q_full = kv_empty + C::kKvStages;     // [stages]
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
  uint64_t* epi_full = s_full + 10;  // d = 64: dK / dV staged in the dS buffer (all compute threads)
  uint64_t* epi_free = s_full + 11;  // d = 64: their stores have read the dS buffer
  uint64_t* dqs_full = s_full + 12;  // d = 64: a dQ partial (or dK / dV) staged (128 arrivals)
  uint64_t* dqs_free = s_full + 13;  // d = 64: the staging buffer is free
  uint64_t* ds_empty2 = s_full + 14;  // second dS buffer (d = 64)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffAbort);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nkt = (N + kTileRows - 1) / kTileRows;
  const int total_units = BH * nkt;
  const int grid = gridDim.x;
  // d = 64 backward: slice-major measured faster at N = 4096 (L2 locality)
  const bool block_major = D == 128 && block_major_order(CAUSAL, total_units, grid, N);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kKvStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&do_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, C::kComputeThreads);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, C::kComputeThreads);
    mbar_init(ds_empty, 1);
    mbar_init(ds_empty2, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, C::kDqWarpgroup ? 128 : C::kComputeThreads);
    mbar_init(dkdv_full, 1);
    mbar_init(dkdv_empty, C::kEpiDqWg ? 128 : C::kComputeThreads);
    mbar_init(mma_done, 1);
    mbar_init(epi_full, C::kComputeThreads);
    mbar_init(epi_free, 1);
    mbar_init(dqs_full, 128);
    mbar_init(dqs_free, 1);
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

  // Each role's code starts with its warpgroup's register budget (d = 128):
  // the warps from the producer on (producer, MMA issuer, idle) give
  // registers back and the compute warpgroups take them.
  if (warp >= C::kComputeWarps) {
    if constexpr (C::kRegSplit) regs_dec<C::kAuxRegs>();
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      Tracer tr(3);
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_do);
      uint32_t ucnt = 0, it = 0;  // K/V copies issued (one per unit, in unit order); Q/dO tiles issued
      bool ok = true;
      // K/V of the unit at `p` into buffer ucnt % kKvStages (waits for the buffer).
      auto issue_kv = [&](int p) -> bool {
        const BwdUnit v = bwd_decode(p, BH, nkt, CAUSAL, block_major);
        const int kb = ucnt % C::kKvStages;
        tr(30);
        if (!mbar_wait(&kv_empty[kb], ((ucnt / C::kKvStages) & 1) ^ 1, status)) return false;
        tr(31);
        mbar_expect_tx(&kv_full[kb], 2 * C::kTileBytes);
        for (int b = 0; b < C::kBlocks; ++b) {
          tma_load_3d(sm + C::kOffK + kb * C::kTileBytes + b * kSwzBlockBytes, &tm_k, &kv_full[kb], b * 64,
                      v.j * kTileRows, v.bh);
          tma_load_3d(sm + C::kOffV + kb * C::kTileBytes + b * kSwzBlockBytes, &tm_v, &kv_full[kb], b * 64,
                      v.j * kTileRows, v.bh);
        }
        ++ucnt;
        return true;
      };
      // Next unit this CTA will process after round r, or -1.
      auto next_pos = [&](int r) -> int {
        for (int rr = r + 1; rr * grid < total_units; ++rr) {
          const int p = snake_unit(rr, blockIdx.x, grid);
          if (p < total_units) return p;
        }
        return -1;
      };
      int prefetched = -1;  // unit whose K/V copy was issued ahead of its turn
      for (int round = 0; ok; ++round) {
        if (round * grid >= total_units) break;
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (pos >= total_units) continue;
        const BwdUnit u = bwd_decode(pos, BH, nkt, CAUSAL, block_major);
        if (prefetched != pos && !(ok = issue_kv(pos))) break;
        prefetched = -1;
        // With two K/V buffers the next unit's copy goes out as soon as its
        // buffer is released: the wait for a Q / dO slot polls that buffer too.
        const int npos = (C::kKvStages > 1) ? next_pos(round) : -1;
        for (int x = 0; x < u.nq && ok; ++x, ++it) {
          const int i = u.qtile(x);
          const int st = it % C::kStages;
          tr(32);
          {
            const uint32_t qa = smem_addr(&qdo_empty[st]);
            const uint32_t qp = ((it / C::kStages) & 1) ^ 1;
            const uint64_t t0 = global_ns();
            while (true) {
              if (npos >= 0 && prefetched < 0 &&
                  mbar_probe(smem_addr(&kv_empty[ucnt % C::kKvStages]), ((ucnt / C::kKvStages) & 1) ^ 1)) {
                if (!(ok = issue_kv(npos))) break;
                prefetched = npos;
              }
              if (mbar_probe(qa, qp)) break;
              if (global_ns() - t0 > kWaitLimitNs) {
                atomicExch(status, kDevTimeout);
                ok = false;
                break;
              }
            }
          }
          tr(33);
          if (!ok) break;
          float* rows = reinterpret_cast<float*>(sm + C::kOffRow + st * C::kRowBytes);
          const size_t roff = (size_t)u.bh * Npad + (size_t)i * kTileRows;
          mbar_expect_tx(&q_full[st], C::kTileBytes + kTileRows * 4);
          for (int b = 0; b < C::kBlocks; ++b)
            tma_load_3d(sm + C::kOffQ + st * C::kTileBytes + b * kSwzBlockBytes, &tm_q, &q_full[st], b * 64,
                        i * kTileRows, u.bh);
          bulk_load_1d(rows, lse2 + roff, kTileRows * 4, &q_full[st]);
          mbar_expect_tx(&do_full[st], C::kTileBytes + kTileRows * 4);
          for (int b = 0; b < C::kBlocks; ++b)
            tma_load_3d(sm + C::kOffDO + st * C::kTileBytes + b * kSwzBlockBytes, &tm_do, &do_full[st], b * 64,
                        i * kTileRows, u.bh);
          bulk_load_1d(rows + kTileRows, dsum + roff, kTileRows * 4, &do_full[st]);
        }
        if (aborted(abort_flag)) ok = false;
      }
      if (!ok) *abort_flag = 1;
      // Drain copies in flight.
      for (uint32_t x = (ucnt > (uint32_t)C::kKvStages ? ucnt - C::kKvStages : 0); x < ucnt; ++x)
        mbar_wait(&kv_full[x % C::kKvStages], (x / C::kKvStages) & 1, status);
      for (uint32_t x = (it > (uint32_t)C::kStages ? it - C::kStages : 0); x < it; ++x) {
        mbar_wait(&q_full[x % C::kStages], (x / C::kStages) & 1, status);
        mbar_wait(&do_full[x % C::kStages], (x / C::kStages) & 1, status);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer --
    {  // whole warp, converged: waits are warp-wide, one elected lane issues
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T: both K-major over d
      const uint32_t idST = kIdSS | s_negate;                  // S^T = (+/-) K Q^T
      constexpr uint32_t kIdKV = idesc_bf16(128, D, 0, 1);    // dV, dK: B (dO / Q) MN-major
      constexpr uint32_t kIdQ = idesc_bf16(128, C::kDqTransposed ? 128 : D, 1, 1);  // dQ / dQ^T: A, B MN-major
      constexpr int kPtRun = C::kQCols / 16;  // 16-query steps with consecutive P^T / dS^T columns
      const uint32_t q_s = smem_addr(sm + C::kOffQ);
      const uint32_t do_s = smem_addr(sm + C::kOffDO);
      const uint32_t ds_s = smem_addr(sm + C::kOffDS);
      uint32_t ucnt = 0, it = 0, pcnt = 0, dscnt = 0, dqcnt = 0;
      bool ok = true;
      Tracer tr(2);
      for (int round = 0; ok; ++round) {
        if (round * grid >= total_units) break;
        const int pos = snake_unit(round, blockIdx.x, grid);
        if (pos >= total_units) continue;
        const BwdUnit u = bwd_decode(pos, BH, nkt, CAUSAL, block_major);
        const int kb = ucnt % C::kKvStages;
        const uint32_t k_s = smem_addr(sm + C::kOffK + kb * C::kTileBytes);
        const uint32_t v_s = smem_addr(sm + C::kOffV + kb * C::kTileBytes);
        auto issue_st = [&](int st) {  // S^T = K Q^T
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)  // four K = 16 steps of 32 bytes per 64-column block
            mma_ss_run_w<4, 2, 2>(tbase + C::kColS, sdesc(k_s + blk * kSwzBlockBytes, 16, 1024),
                                  sdesc(q_s + st * C::kTileBytes + blk * kSwzBlockBytes, 16, 1024), idST, blk > 0);
          mma_commit_w(s_full);
        };
        auto issue_dp = [&](int st) {  // dP^T = V dO^T
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            mma_ss_run_w<4, 2, 2>(tbase + C::kColDP, sdesc(v_s + blk * kSwzBlockBytes, 16, 1024),
                                  sdesc(do_s + st * C::kTileBytes + blk * kSwzBlockBytes, 16, 1024), kIdSS, blk > 0);
          mma_commit_w(dp_full);
        };
        tr(10);
        ok = mbar_wait_warp(&kv_full[kb], (ucnt / C::kKvStages) & 1, status);
        tr(11);
        if (!ok) break;
        {
          const int st = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          ok = mbar_wait_warp(&q_full[st], ph, status);
          if (!ok) break;
          tc_fence_after();
          issue_st(st);
          if (C::kEarlyDp) {
            ok = mbar_wait_warp(&do_full[st], ph, status);
            if (!ok) break;
            tc_fence_after();
            issue_dp(st);
          }
        }
        for (int x = 0; x < u.nq && ok; ++x, ++it) {
          const int st = it % C::kStages;
          const int st2 = (it + 1) % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          const uint32_t ph2 = ((it + 1) / C::kStages) & 1;
          if (!C::kEarlyDp) {
            // dP^T(i) once dO(i) is in and the dQ^T partial sharing its columns is drained
            tr(12);
            ok = mbar_wait_warp(&do_full[st], ph, status);
            if (ok) ok = mbar_wait_warp(dq_empty, (dqcnt & 1) ^ 1, status);
            tr(18);
            if (!ok) break;
            tc_fence_after();
            issue_dp(st);
            tr(13);
          }
          // dV += P^T dO  (A = P^T from TMEM, B = dO MN-major); the first of a unit
          // also waits until the previous unit's dK/dV have been read out.
          ok = mbar_wait_warp(p_full, pcnt & 1, status);
          if (ok && x == 0) ok = mbar_wait_warp(dkdv_empty, (ucnt & 1) ^ 1, status);
          tr(14);
          ++pcnt;
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int r = 0; r < kTileRows / 16 / kPtRun; ++r)  // runs of kPtRun 16-query steps (pt_col)
            mma_ts_run_w<kPtRun, 8, 128>(tbase + C::kColDV, tbase + C::kColS + pt_col<C::kQCols>(r * kPtRun),
                                         sdesc(do_s + st * C::kTileBytes + r * kPtRun * 2048, kSwzBlockBytes, 1024),
                                         kIdKV, (x > 0 || r > 0));
          tr(19);
          // S^T(i+1) as early as possible
          if (x + 1 < u.nq) {
            ok = mbar_wait_warp(&q_full[st2], ph2, status);
            tr(20);
            if (!ok) break;
            tc_fence_after();
            issue_st(st2);
          }
          // dS(i) in shared memory: dK += dS^T Q (then the Q / dO slot is
          // free: Q(i) has no later reader), [dP^T(i+1)], dQ_part = dS K
          tr(15);
          ok = mbar_wait_warp(ds_full, dscnt & 1, status);
          const int db = dscnt % C::kDsBufs;
          ++dscnt;
          if (!ok) break;
          tc_fence_after();
          const uint32_t dsb = ds_s + db * C::kDsBytes;
          if constexpr (C::kDsTmem) {  // dK += dS^T Q, dS^T packed over the dP^T columns
#pragma unroll
            for (int r = 0; r < kTileRows / 16 / kPtRun; ++r)
              mma_ts_run_w<kPtRun, 8, 128>(tbase + C::kColDK, tbase + C::kColDP + pt_col<C::kQCols>(r * kPtRun),
                                           sdesc(q_s + st * C::kTileBytes + r * kPtRun * 2048, kSwzBlockBytes, 1024),
                                           kIdKV, (x > 0 || r > 0));
          } else {
#pragma unroll
            for (int blk = 0; blk < kTileRows / 64; ++blk)  // dS^T K-major: 32-byte steps in a block; Q: 16 rows
              mma_ss_run_w<4, 2, 128>(tbase + C::kColDK, sdesc(dsb + blk * kSwzBlockBytes, 16, 1024),
                                      sdesc(q_s + st * C::kTileBytes + blk * 4 * 2048, kSwzBlockBytes, 1024), kIdKV,
                                      (x > 0 || blk > 0));
          }
          mma_commit_w(&qdo_empty[st]);  // Q(i), dO(i) read for the last time: the producer may reload the slot
          if (C::kEarlyDp && x + 1 < u.nq) {
            tr(12);
            ok = mbar_wait_warp(&do_full[st2], ph2, status);
            tr(18);
            if (!ok) break;
            tc_fence_after();
            issue_dp(st2);
            tr(13);
          }
          if (DQ && !C::kDqAliasesDp) ok = mbar_wait_warp(dq_empty, (dqcnt & 1) ^ 1, status);
          tr(16);
          if (!ok) break;
          tc_fence_after();
          if (DQ) {
            const uint64_t dsd = sdesc(dsb, kSwzBlockBytes, 1024);  // dS^T, 16 keys (2048 bytes) a step
            const uint64_t kd = sdesc(k_s, kSwzBlockBytes, 1024);   // K, 16 keys a step
            if (C::kDqTransposed)
              mma_ss_run_w<8, 128, 128>(tbase + C::kColDQ, kd, dsd, kIdQ, 0);  // dQ^T = K^T dS^T
            else
              mma_ss_run_w<8, 128, 128>(tbase + C::kColDQ, dsd, kd, kIdQ, 0);  // dQ = dS K
            mma_commit_w(dq_full);
          }
          mma_commit_w(db ? ds_empty2 : ds_empty);
          ++dqcnt;
          tr(17);
        }
        if (!ok) break;
        mma_commit_w(dkdv_full);
        mma_commit_w(&kv_empty[kb]);
        ++ucnt;
        if (__any_sync(0xffffffffu, aborted(abort_flag))) ok = false;
      }
      if (!ok) *abort_flag = 1;
      mma_commit_w(mma_done);
      mbar_wait_warp(mma_done, 0, status);
    }
  } else if (C::kDqWarpgroup) {
    // ----------------------------------------------------- dQ warpgroup --
    // d = 64 only: thread = query row r; it reads its 64-column dQ row, releases
    // the columns, writes the row into a pair of 128-byte-swizzled 32-column
    // boxes, and one thread issues the tensor reduce-adds.
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const uint32_t t_dq = tmem_lane_col(tbase, quarter * 32, C::kColDQ);
    const bool elected = (warp == C::kDqWarp0) && (lane == 0);
    uint32_t qcnt = 0;  // dQ partials drained
    uint32_t stg = 0;   // uses of the staging buffer (dQ partials and dK / dV)
    uint32_t ucnt = 0;  // units whose dK / dV this warpgroup wrote
    bool ok = true;
    Tracer tr(warp == C::kDqWarp0 + 2 ? 1 : -1);
    for (int round = 0; ok; ++round) {
      if (round * grid >= total_units) break;
      const int pos = snake_unit(round, blockIdx.x, grid);
      if (pos >= total_units) continue;
      const BwdUnit u = bwd_decode(pos, BH, nkt, CAUSAL, block_major);
      for (int x = 0; x < u.nq && ok; ++x) {
        tr(40);
        ok = mbar_wait_warp(dq_full, qcnt & 1, status);
        ++qcnt;
        if (!ok) break;
        tc_fence_after();
        {
          uint8_t* stage = sm + C::kOffDQS;
          if (elected) {
            tma_store_wait_read0();  // the previous reduce-adds have read the buffer
            mbar_arrive(dqs_free);
          }
          if (!(ok = mbar_wait_warp(dqs_free, stg & 1, status))) break;
          // Both 32-column halves at once; with 4 compute warpgroups (fewer
          // registers per thread) one half at a time.
          constexpr int kHalvesAtOnce = (C::kWG == 4) ? 1 : 2;
          const int swz = r & 7;
#pragma unroll
          for (int b0 = 0; b0 < 2; b0 += kHalvesAtOnce) {
            uint32_t v[32 * kHalvesAtOnce];
#pragma unroll
            for (int h = 0; h < kHalvesAtOnce; ++h)
              tmem_ld32(t_dq + 32 * (b0 + h), *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
            tmem_wait_ld();
            if (b0 + kHalvesAtOnce == 2) {  // the whole row is read: release the columns
              tc_fence_before();
              mbar_arrive(dq_empty);
              tr(41);
            }
#pragma unroll
            for (int h = 0; h < kHalvesAtOnce; ++h)
#pragma unroll
              for (int m = 0; m < 8; ++m)
                *reinterpret_cast<uint4*>(stage + (b0 + h) * (C::kDqStageBytes / 2) + r * 128 + ((m ^ swz) * 16)) =
                    make_uint4(v[32 * h + 4 * m], v[32 * h + 4 * m + 1], v[32 * h + 4 * m + 2],
                               v[32 * h + 4 * m + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(dqs_full);
          if (warp == C::kDqWarp0) {
            if (!(ok = mbar_wait_warp(dqs_full, stg & 1, status))) break;
            if (lane == 0) {
              for (int b = 0; b < 2; ++b)
                tma_reduce_add_3d(&tm_dqacc, stage + b * (C::kDqStageBytes / 2), 32 * b, u.qtile(x) * kTileRows,
                                  u.bh);
              tma_store_commit();
            }
          }
          ++stg;
        }
        tr(42);
      }
      if (!ok) break;
      if constexpr (C::kEpiDqWg) {
        // ---- the unit's dV and dK (x scale) -> bf16 -> two TMA stores ----
        // Thread r holds key row r: its 64 dV columns go to box 0 of the
        // staging buffer, its dK columns to box 1 (128-byte-swizzled 64-column
        // boxes, chunk m of row r at m ^ (r % 8)).  Rows past N are clipped.
        ok = mbar_wait_warp(dkdv_full, ucnt & 1, status);
        ++ucnt;
        if (!ok) break;
        tc_fence_after();
        uint8_t* stage = sm + C::kOffDQS;
        if (elected) {
          tma_store_wait_read0();  // the last reduce-adds have read the buffer
          mbar_arrive(dqs_free);
        }
        if (!(ok = mbar_wait_warp(dqs_free, stg & 1, status))) break;
        const int swz = r & 7;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // 0: dV, 1: dK
          uint32_t v[64];
          const uint32_t t_acc = tmem_lane_col(tbase, quarter * 32, h ? C::kColDK : C::kColDV);
          tmem_ld32(t_acc, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(t_acc + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          if (h == 1) {  // both accumulators read: the next unit may overwrite them
            tc_fence_before();
            mbar_arrive(dkdv_empty);
          }
          const float sc = h ? scale : 1.f;
          uint8_t* row = stage + h * (C::kDqStageBytes / 2) + r * 128;
#pragma unroll
          for (int m = 0; m < 8; ++m)
            *reinterpret_cast<uint4*>(row + ((m ^ swz) * 16)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * m]) * sc, __uint_as_float(v[8 * m + 1]) * sc),
                           pack_bf16x2(__uint_as_float(v[8 * m + 2]) * sc, __uint_as_float(v[8 * m + 3]) * sc),
                           pack_bf16x2(__uint_as_float(v[8 * m + 4]) * sc, __uint_as_float(v[8 * m + 5]) * sc),
                           pack_bf16x2(__uint_as_float(v[8 * m + 6]) * sc, __uint_as_float(v[8 * m + 7]) * sc));
        }
        fence_proxy_async_smem();
        mbar_arrive(dqs_full);
        if (warp == C::kDqWarp0) {
          if (!(ok = mbar_wait_warp(dqs_full, stg & 1, status))) break;
          if (lane == 0) {
            tma_store_3d(&tm_dv, stage, 0, u.j * kTileRows, u.bh);
            tma_store_3d(&tm_dk, stage + C::kDqStageBytes / 2, 0, u.j * kTileRows, u.bh);
            tma_store_commit();
          }
        }
        ++stg;
      }
      if (aborted(abort_flag)) ok = false;
    }
    if (!ok) *abort_flag = 1;
    if (elected) tma_store_wait_all0();  // reductions in flight land before the CTA exits
    }
  } else {
    if constexpr (C::kRegSplit) regs_inc<C::kComputeRegs>();
    // ------------------------------------------------ compute warpgroups --
    // Warpgroup g owns query columns [kQCols g, kQCols (g+1)) of P^T / dS^T
    // (and of the dQ^T partial at d = 128), and columns [kDCols g,
    // kDCols (g+1)) of dV and dK.
    constexpr int kQC = C::kQCols;
    constexpr int kDC = C::kDCols;
    const int g = warp / 4;
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;  // key row (P, dS, dK, dV) / head-dimension row (dQ^T) in the tile
    const uint32_t lanes = (uint32_t)quarter * 32;
    const uint32_t t_s = tmem_lane_col(tbase, lanes, C::kColS + kQC * g);
    const uint32_t t_dp = tmem_lane_col(tbase, lanes, C::kColDP + kQC * g);
    const uint32_t t_dq = tmem_lane_col(tbase, lanes, C::kColDQ + kQC * g);
    const uint32_t t_dv = tmem_lane_col(tbase, lanes, C::kColDV + kDC * g);
    const uint32_t t_dk = tmem_lane_col(tbase, lanes, C::kColDK + kDC * g);
    // dS^T row r in shared memory: query q is 16-byte chunk q / 8 of the row,
    // in swizzle block (q / 8) / 8 at position (q / 8) % 8.
    const int chunk0 = kQC * g / 8;
    uint8_t* ds_row0 = sm + C::kOffDS + (chunk0 / 8) * kSwzBlockBytes + r * 128;  // + buffer * kDsBytes
    const int cbase = chunk0 % 8;
    const int swz = r & 7;
    const uint64_t c2x2 = f2_pack(c2, c2);
    uint32_t scnt = 0, dpcnt = 0, dse = 0, ucnt = 0, qit = 0, dqcnt = 0;
    uint32_t ecnt = 0;        // d = 64: units whose dK / dV went out through the dS buffer
    bool epi_pending = false;  // ... the last of which may still be reading it
    int pend_bh = 0, pend_qt = -1;  // dQ partial still to drain from the previous unit
    // (not with dropout: its keep bits leave no registers for the held values)
    constexpr bool kDqInterleave = C::kDqTransposed && !DROP;
    constexpr int kDqNow = kBwdDqImmediate < kQC ? kBwdDqImmediate : kQC;
    constexpr int kDqPerChunk = (kQC - kDqNow) / (kQC / 8);  // the dS loop has kQC / 8 chunks
    static_assert(!kDqInterleave || kDqNow + kDqPerChunk * (kQC / 8) == kQC, "dQ reductions split");

    bool ok = true;
    Tracer tr(warp == 0 ? 0 : -1);

    // Read this warpgroup's half of the dQ^T partial of query tile `qt` from
    // TMEM, release the columns, then add it into the fp32 accumulator (d = 128
    // unless the dedicated dQ warpgroup drains it).
    auto drain_dq = [&](int bh, int qt) -> bool {
      tr(40);
      if (!mbar_wait_warp(dq_full, dqcnt & 1, status)) return false;
      ++dqcnt;
      tc_fence_after();
      if (C::kDqTransposed) {
        // lane = head-dimension index r, columns = this warpgroup's queries:
        // one scalar reduction per query, 128 contiguous bytes per warp.
        uint32_t v[kQC];
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c) tmem_ld32(t_dq + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(dq_empty);
        tr(41);
        const int q0 = qt * kTileRows + kQC * g;
        float* dst = dq_acc + ((size_t)bh * N + q0) * D + r;
        const int nvalid = N - q0;
#pragma unroll
        for (int c = 0; c < kQC; ++c)
          if (c < nvalid) red_add(dst + (size_t)c * D, __uint_as_float(v[c]));
      }
      return true;
    };

    for (int round = 0; ok; ++round) {
      if (round * grid >= total_units) break;
      const int pos = snake_unit(round, blockIdx.x, grid);
      if (pos >= total_units) continue;
      const BwdUnit u = bwd_decode(pos, BH, nkt, CAUSAL, block_major);
      const int kr = u.j * kTileRows + r;  // this thread's key
      const bool key_ok = kr < N;
      for (int x = 0; x < u.nq; ++x, ++qit) {
        const int i = u.qtile(x);
        const int qbase = i * kTileRows + kQC * g;  // first query of this warpgroup's columns
        const bool diag = CAUSAL && (i == u.j);
        // -lse2 / -D of this query tile, staged in shared memory with Q / dO
        const float* rows =
            reinterpret_cast<const float*>(sm + C::kOffRow + (qit % C::kStages) * C::kRowBytes) + kQC * g;
        // ---- P^T = 2^(S^T c2 - lse2); masked entries exactly 0 ----
        tr(1);
        ok = mbar_wait_warp(s_full, scnt & 1, status);
        tr(2);
        ++scnt;
        if (!ok) break;
        tc_fence_after();
        uint32_t pk[kQC / 2];  // this warpgroup's P^T row, bf16 pairs (reused for dS)
        uint32_t svall[kQC];   // the whole S^T row piece: every load in flight, one wait
        // DROP: keep bit of (query qbase + c, this thread's key) for c < kQC.  A
        // generator call covers four consecutive keys, which sit in four
        // consecutive lanes: lane s of a group computes the call for query
        // qb + s and the group exchanges words in three shuffles, so that
        // each lane ends with its own key's word for the four queries.
        uint64_t keep = ~0ull;
        if (DROP) {
          keep = 0ull;
          const int s4 = lane & 3, g4 = lane & ~3;
#pragma unroll 4
          for (int b4 = 0; b4 < kQC / 4; ++b4) {
            const uint4 w = philox4x32_10((uint32_t)(kr >> 2), (uint32_t)(qbase + 4 * b4 + s4), (uint32_t)u.bh,
                                          dp.offset, dp.k0, dp.k1);
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int want = (s4 - rr) & 3;  // the word the lane reading from this one needs
              const uint32_t val = want == 0 ? w.x : want == 1 ? w.y : want == 2 ? w.z : w.w;
              const uint32_t got = __shfl_sync(0xffffffffu, val, g4 | ((s4 + rr) & 3));
              if (got >= dp.thr) keep |= 1ull << (4 * b4 + ((s4 + rr) & 3));
            }
          }
        }
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c) tmem_ld32(t_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&svall[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c) {
          const uint32_t* sv = svall + 32 * c;
          // -lse2 of the 32 queries, four per 16-byte broadcast load
          ulonglong2 nlv[8];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) nlv[e4] = *reinterpret_cast<const ulonglong2*>(rows + 32 * c + 4 * e4);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t nl2 = (e & 1) ? nlv[e / 2].y : nlv[e / 2].x;
            const uint64_t xx = f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), c2x2, nl2);
            float x0, x1;
            f2_unpack(xx, x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if (diag) {
              const int q = qbase + 32 * c + 2 * e;
              if (q < kr) p0 = 0.f;
              if (q + 1 < kr) p1 = 0.f;
            }
            pk[16 * c + e] = key_ok ? pack_bf16x2(p0, p1) : 0u;
          }
          if (DROP) {  // the dV operand: surviving probabilities times 1 / (1 - p), over this chunk's S^T columns
            uint32_t pt[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[16 * c + e]));
              const int bit = 32 * c + 2 * e;
              pt[e] = pack_bf16x2(((keep >> bit) & 1) ? pf.x * dp.inv_keep : 0.f,
                                  ((keep >> (bit + 1)) & 1) ? pf.y * dp.inv_keep : 0.f);
            }
            tmem_st16(t_s + 16 * c, pt);
          }
        }
        // This warpgroup's S^T columns are fully read: P^T goes over the first half.
        if (!DROP) {
#pragma unroll
          for (int c = 0; c < kQC / 32; ++c) tmem_st16(t_s + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * c]));
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
        tr(3);
        // ---- dQ partial of the previous query tile ----
        // d = 128 (without dropout): the drained dQ^T column piece
        // waiting for its reductions (issued by this tile's dS loop)
        uint32_t dqv[kDqInterleave ? kQC : 1];
        float* dq_dst = dq_acc;
        int dq_nvalid = 0;
        bool dq_have = false;
        if (DQ && !C::kDqWarpgroup) {
          // dQ of the previous query tile: this unit's, or the last one of
          // the previous unit (deferred so the unit boundary does not wait).
          int dbh = -1, dqt = 0;  // the partial to drain, if any
          if (x > 0) {
            dbh = u.bh;
            dqt = u.qtile(x - 1);
          } else if (pend_qt >= 0) {
            dbh = pend_bh;
            dqt = pend_qt;
            pend_qt = -1;
          }
          if (dbh >= 0) {
            if constexpr (kDqInterleave) {
              // read this warpgroup's dQ^T columns and release them; the
              // reductions go out with the dS loop below
              tr(40);
              ok = mbar_wait_warp(dq_full, dqcnt & 1, status);
              ++dqcnt;
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int c = 0; c < kQC / 32; ++c)
                tmem_ld32(t_dq + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&dqv[32 * c]));
              tmem_wait_ld();
              tc_fence_before();
              mbar_arrive(dq_empty);
              tr(41);
              const int q0 = dqt * kTileRows + kQC * g;
              dq_dst = dq_acc + ((size_t)dbh * N + q0) * D + r;
              dq_nvalid = N - q0;
              dq_have = true;
              // the first kDqNow now (fewer values live through the dS loop)
#pragma unroll
              for (int c = 0; c < kDqNow; ++c)
                if (c < dq_nvalid) red_add(dq_dst + (size_t)c * D, __uint_as_float(dqv[c]));
            } else {
              if (!(ok = drain_dq(dbh, dqt))) break;
            }
          }
        }
        // ---- dS^T = P^T (dP^T - D) -> shared memory (bf16, swizzled) ----
        tr(42);
        ok = mbar_wait_warp(dp_full, dpcnt & 1, status);
        tr(43);
        ++dpcnt;
        const int db = dse % C::kDsBufs;
        if (ok) ok = mbar_wait_warp(db ? ds_empty2 : ds_empty, ((dse / C::kDsBufs) & 1) ^ 1, status);
        ++dse;
        uint8_t* ds_row = ds_row0 + db * C::kDsBytes;
        if (ok && C::kEpiTma && !C::kEpiDqWg && epi_pending) {  // the previous unit's dK / dV stores read the buffer
          if (warp == 0 && lane == 0) {
            tma_store_wait_read0();
            mbar_arrive(epi_free);
          }
          ok = mbar_wait_warp(epi_free, (ecnt - 1) & 1, status);
          epi_pending = false;
        }
        tr(4);
        if (!ok) break;
        tc_fence_after();
        uint32_t dpall[kQC];  // the whole dP^T row piece: every load in flight, one wait
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c) tmem_ld32(t_dp + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&dpall[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c) {
          const uint32_t* dpv = dpall + 32 * c;
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {  // four 16-byte chunks = 32 queries
            const int m = 4 * c + mm;
            uint32_t dsk[4];
            // -D of the chunk's 8 queries, four per 16-byte broadcast load
            const ulonglong2 nd01 = *reinterpret_cast<const ulonglong2*>(rows + kTileRows + 8 * m);
            const ulonglong2 nd23 = *reinterpret_cast<const ulonglong2*>(rows + kTileRows + 8 * m + 4);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int idx = 4 * m + e;  // pair index within the half
              const uint64_t nd = (e == 0) ? nd01.x : (e == 1) ? nd01.y : (e == 2) ? nd23.x : nd23.y;
              const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[idx]));
              float dp0 = __uint_as_float(dpv[8 * mm + 2 * e]), dp1 = __uint_as_float(dpv[8 * mm + 2 * e + 1]);
              if (DROP) {  // dP o M / (1 - p)
                const int bit = 2 * idx;
                dp0 = ((keep >> bit) & 1) ? dp0 * dp.inv_keep : 0.f;
                dp1 = ((keep >> (bit + 1)) & 1) ? dp1 * dp.inv_keep : 0.f;
              }
              const uint64_t t = f2_add(f2_pack(dp0, dp1), nd);
              float d0, d1;
              f2_unpack(f2_mul(f2_pack(pf.x, pf.y), t), d0, d1);
              dsk[e] = pack_bf16x2(d0, d1);
            }
            if constexpr (C::kDsTmem) {  // P^T is no longer needed: its registers keep dS^T for tensor memory
#pragma unroll
              for (int e = 0; e < 4; ++e) pk[4 * m + e] = dsk[e];
            }
            if constexpr (C::kDsSmem)
              *reinterpret_cast<uint4*>(ds_row + (((cbase + m) ^ swz) * 16)) =
                  make_uint4(dsk[0], dsk[1], dsk[2], dsk[3]);
            if (kDqInterleave && dq_have) {  // the rest, kDqPerChunk per chunk of eight queries
#pragma unroll
              for (int e4 = 0; e4 < kDqPerChunk; ++e4) {
                const int c = kDqNow + kDqPerChunk * m + e4;
                if (c < dq_nvalid) red_add(dq_dst + (size_t)c * D, __uint_as_float(dqv[c]));
              }
            }
          }
        }
        if constexpr (C::kDsTmem) {
#pragma unroll
          for (int c = 0; c < kQC / 32; ++c) tmem_st16(t_dp + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * c]));
          tmem_wait_st();
        }
        if constexpr (C::kDsSmem) fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ds_full);
        tr(5);
      }
      if (!ok) break;
      // ---- dQ partial of the unit's last query tile ----
      if (DQ && !C::kDqWarpgroup) {  // the unit's last dQ partial drains after P(0) of the next unit
        pend_bh = u.bh;
        pend_qt = u.qtile(u.nq - 1);
      }
      // ---- epilogue: this warpgroup's half of the dV, dK (x scale) columns -> bf16 ----
      // (with the dQ warpgroup, that warpgroup writes them)
      if constexpr (C::kEpiDqWg) {
        if (aborted(abort_flag)) ok = false;
        continue;
      }
      tr(6);
      ok = mbar_wait_warp(dkdv_full, ucnt & 1, status);
      ++ucnt;
      if (!ok) break;
      tc_fence_after();
      if (C::kEpiTma) {
        // dV, dK (x scale) -> bf16 in the dS buffer as 128-byte-swizzled
        // 64-column boxes (block 0 dV, block 1 dK; this warpgroup writes
        // columns [kDCols g, kDCols (g+1)) of its key row), then one thread
        // stores both boxes.  Rows past N are clipped by the copy.
        uint32_t a[kDC], b[kDC];
#pragma unroll
        for (int c = 0; c < kDC / 16; ++c) {
          tmem_ld16(t_dv + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&a[16 * c]));
          tmem_ld16(t_dk + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&b[16 * c]));
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(dkdv_empty);  // the next unit may overwrite the columns
        uint8_t* rv = sm + C::kOffDS + r * 128;
        uint8_t* rk = rv + kSwzBlockBytes;
#pragma unroll
        for (int m = 0; m < kDC / 8; ++m) {
          const int ch = ((kDC * g / 8 + m) ^ swz) * 16;
          *reinterpret_cast<uint4*>(rv + ch) =
              make_uint4(pack_bf16x2(__uint_as_float(a[8 * m]), __uint_as_float(a[8 * m + 1])),
                         pack_bf16x2(__uint_as_float(a[8 * m + 2]), __uint_as_float(a[8 * m + 3])),
                         pack_bf16x2(__uint_as_float(a[8 * m + 4]), __uint_as_float(a[8 * m + 5])),
                         pack_bf16x2(__uint_as_float(a[8 * m + 6]), __uint_as_float(a[8 * m + 7])));
          *reinterpret_cast<uint4*>(rk + ch) =
              make_uint4(pack_bf16x2(__uint_as_float(b[8 * m]) * scale, __uint_as_float(b[8 * m + 1]) * scale),
                         pack_bf16x2(__uint_as_float(b[8 * m + 2]) * scale, __uint_as_float(b[8 * m + 3]) * scale),
                         pack_bf16x2(__uint_as_float(b[8 * m + 4]) * scale, __uint_as_float(b[8 * m + 5]) * scale),
                         pack_bf16x2(__uint_as_float(b[8 * m + 6]) * scale, __uint_as_float(b[8 * m + 7]) * scale));
        }
        fence_proxy_async_smem();
        mbar_arrive(epi_full);
        if (warp == 0) {
          ok = mbar_wait_warp(epi_full, ecnt & 1, status);
          if (ok && lane == 0) {
            tma_store_3d(&tm_dv, sm + C::kOffDS, 0, u.j * kTileRows, u.bh);
            tma_store_3d(&tm_dk, sm + C::kOffDS + kSwzBlockBytes, 0, u.j * kTileRows, u.bh);
            tma_store_commit();
          }
        }
        ++ecnt;
        epi_pending = true;
        if (!ok) break;
      } else {
        // Each thread stores its key row's kDCols columns of dV and dK.
        const size_t rowoff = ((size_t)u.bh * N + kr) * D + kDC * g;
#pragma unroll
        for (int c = 0; c < kDC / 32; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32(t_dv + 32 * c, a);
          tmem_ld32(t_dk + 32 * c, b);
          tmem_wait_ld();
          if (c == kDC / 32 - 1) {  // dK / dV columns read: the next unit may overwrite them
            tc_fence_before();
            mbar_arrive(dkdv_empty);
          }
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
      }
      tr(7);
      if (aborted(abort_flag)) ok = false;
    }
    if (DQ && ok && pend_qt >= 0) ok = drain_dq(pend_bh, pend_qt);  // reduced at once: no dS loop follows
    if (!ok) *abort_flag = 1;
    // dK / dV stores still in flight must finish before the CTA exits.
    if (C::kEpiTma && !C::kEpiDqWg && warp == 0 && lane == 0) tma_store_wait_all0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool DQ, bool DROP = false>
static cudaError_t launch_main_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = BwdCfg<D, DQ>;
  auto kern = fa_bwd_main<D, CAUSAL, DQ, DROP>;
  if constexpr (C::kRegSplit) {
    // The register split assumes a build at exactly kLaunchRegs registers a
    // thread: with fewer, the compute warpgroups' request could never be met.
    static const bool regs_ok = [&] {
      cudaFuncAttributes fa_attr;
      return cudaFuncGetAttributes(&fa_attr, kern) == cudaSuccess && fa_attr.numRegs == C::kLaunchRegs;
    }();
    if (!regs_ok) return cudaErrorInvalidKernelImage;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, C::kThreads, C::kSmemBytes, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dqacc, *a.tm_dk,
                                                       *a.tm_dv, a.lse2,
                                                       a.dsum, a.dq_acc, reinterpret_cast<__nv_bfloat16*>(a.dk),
                                                       reinterpret_cast<__nv_bfloat16*>(a.dv), a.BH, a.N, a.Npad,
                                                       a.c2, a.scale, a.drop, a.status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t stream) {
  auto o = reinterpret_cast<const __nv_bfloat16*>(a.o);
  auto dout = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  if (a.d == 64)
    fa_bwd_pre<64><<<a.pre_grid, 256, 0, stream>>>(o, dout, a.lse, a.lse2, a.dsum, a.dq_acc, a.BH, a.N, a.Npad,
                                                   a.with_dq);
  else
    fa_bwd_pre<128><<<a.pre_grid, 256, 0, stream>>>(o, dout, a.lse, a.lse2, a.dsum, a.dq_acc, a.BH, a.N, a.Npad,
                                                    a.with_dq);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdLaunch& a, cudaStream_t stream) {
  if (a.dropout) {  // the fused backward only
    if (a.d == 64)
      return a.causal ? launch_main_t<64, true, true, true>(a, stream) : launch_main_t<64, false, true, true>(a, stream);
    return a.causal ? launch_main_t<128, true, true, true>(a, stream) : launch_main_t<128, false, true, true>(a, stream);
  }
  if (a.with_dq) {
    if (a.d == 64) return a.causal ? launch_main_t<64, true, true>(a, stream) : launch_main_t<64, false, true>(a, stream);
    return a.causal ? launch_main_t<128, true, true>(a, stream) : launch_main_t<128, false, true>(a, stream);
  }
  if (a.d == 64) return a.causal ? launch_main_t<64, true, false>(a, stream) : launch_main_t<64, false, false>(a, stream);
  return a.causal ? launch_main_t<128, true, false>(a, stream) : launch_main_t<128, false, false>(a, stream);
}

cudaError_t launch_bwd_conv(const BwdLaunch& a, cudaStream_t stream) {
  const long long n8 = (long long)a.BH * a.N * a.d / 8;
  fa_bwd_dq_conv<<<a.pre_grid, 256, 0, stream>>>(a.dq_acc, reinterpret_cast<__nv_bfloat16*>(a.dq), n8, a.scale);
  return cudaGetLastError();
}

int bwd_units(int BH, int N) { return BH * ((N + kTileRows - 1) / kTileRows); }

}  // namespace fa

#ifdef FA_TRACE
// Trace builds only: phase records of this file's kernels.
extern "C" int fa_trace_dump_bwd(void* host, size_t bytes) { return fa::trace_dump(host, bytes); }
#endif
