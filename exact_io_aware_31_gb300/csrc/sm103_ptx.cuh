// Thin inline-PTX layer for sm_103a: mbarriers with bounded waits, TMA tile
// copies, and the tcgen05 tensor-core family (TMEM allocation, MMA issue,
// commit, TMEM loads/stores) plus the shared-memory and instruction descriptors
// those MMAs consume.  Written from the public PTX ISA description of these
// instructions; nothing here depends on CUTLASS.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace fa {

// ---------------------------------------------------------------- errors ----
// Device status codes written into the library's status word (see fa.h).
enum : int {
  kDevOk = 0,
  kDevTimeout = 5,   // FA_ERR_DEVICE_TIMEOUT
  kDevInternal = 6,  // FA_ERR_INTERNAL
};

// Shared-memory tiles are laid out from the dynamic shared memory base, which
// must be 1024-byte aligned for the 128-byte swizzle atoms.  On sm_103 the
// base follows the 1 KiB reserved block and is 1024-aligned; a kernel that
// finds otherwise records kDevInternal and returns before touching memory.
__device__ __forceinline__ bool smem_base_ok(const void* base, int* status) {
  if ((static_cast<uint32_t>(__cvta_generic_to_shared(base)) & 1023u) == 0) return true;
  if (threadIdx.x == 0) atomicExch(status, kDevInternal);
  return false;
}

// Every mbarrier wait gives up after this many nanoseconds of global time,
// records kDevTimeout and lets the CTA leave cleanly.  Legitimate waits in
// these kernels last microseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarriers ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_probe(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (after recording kDevTimeout in *status) if it has not within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  const uint32_t a = smem_addr(bar);
  if (mbar_test(a, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_test(a, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicExch(status, kDevTimeout);
      return false;
    }
  }
}

// Warp-uniform wait: every lane tests the barrier itself (acquire) and the warp
// leaves together once all lanes have seen the phase complete, so the fast
// path costs one test and one vote.  The time limit is checked by lane 0 and
// broadcast, so a timeout is also warp-uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* status) {
  const uint32_t a = smem_addr(bar);
  bool done = mbar_test(a, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i) {
      done = done || mbar_test(a, parity);
      if (__all_sync(0xffffffffu, done)) return true;
    }
    const bool expired = __shfl_sync(0xffffffffu, (global_ns() - t0 > kWaitLimitNs) ? 1 : 0, 0) != 0;
    if (expired) {
      if ((threadIdx.x & 31) == 0) atomicExch(status, kDevTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------ register budgets ----
// Move this warpgroup's per-thread register budget up or down (all four warps
// of the warpgroup execute it).  The registers a warpgroup gives back go to
// the others of the block; the block's total is what it was launched with, so
// the budgets a kernel sets must add up to no more than that total.
template <int N>
__device__ __forceinline__ void regs_inc() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "register budget");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "register budget");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ fences --
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier among `nthreads` threads (multiple of 32) of this CTA.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// -------------------------------------------------------------------- TMA ---
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled store shared -> global (out-of-range rows are clipped by the unit).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
      : "memory");
}

// 3-D tiled reduce-add shared -> global (fp32 add; out-of-range rows clipped).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
      : "memory");
}

// Wait until at most one committed bulk group still reads shared memory.
__device__ __forceinline__ void tma_store_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the smem sources of all committed stores have been read.
__device__ __forceinline__ void tma_store_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until all committed stores are complete (visible in global memory).
__device__ __forceinline__ void tma_store_wait_all0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------- thread-block clusters ---
// Every thread of every CTA of the cluster arrives (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// fp32 at this CTA's shared address `addr`, as seen in cluster CTA `rank`.
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr, int rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// ---------------------------------------------------------------- tcgen05 ---
// TMEM address: bits 31..16 lane, bits 15..0 column (32-bit columns).
__device__ __forceinline__ uint32_t tmem_lane_col(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// Whole warp: allocate `ncols` TMEM columns, address written to *dst (smem).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// tcgen05.mma kind::f16 on one CTA, D in TMEM: mma_ss takes A and B from
// shared memory descriptors, mma_ts takes A from TMEM; mma_commit_w arrives
// once on `bar` when every tcgen05 op the issuing lane started is done.
// Warp-collective issue: the whole warp calls these, converged, and the lane
// that elect.sync picks (the lowest active lane, so always lane 0 of a full
// warp) issues.  Measured on GB300, one lane issuing from inside a divergent
// branch costs far more issue slots per MMA than this form: a stream of
// 128x64x16 MMAs ran 1.4x slower on an idle sub-partition and 2.2x slower when
// two ALU-bound warps shared it.  A commit issued this way tracks the MMAs
// issued this way (same lane).
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 t;\n\telect.sync t|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 t;\n\telect.sync t|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Runs of kind::f16 MMAs into one accumulator under a single elect.sync: the
// k-th MMA of a run of NK (2, 4 or 8) takes the A and B operands advanced by
// k steps (descriptor steps in 16-byte units, added to the start-address
// field; a TMEM A step in columns).  The first MMA accumulates when
// `accumulate` is set, the others always.  One election and one predicate
// for the run, and descriptor steps as adds, instead of the full single-MMA
// sequence each: measured on GB300, the MMA warp shares its sub-partition
// with busy softmax or compute warps, and the d = 64 forward on the GPT-2
// shape ran 7% faster with its MMAs issued this way.
#define FA_RUN_HEAD                                                                                   \
  "{\n\t.reg .pred p, e, q;\n\t.reg .b32 t;\n\t.reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"              \
  "elect.sync t|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %3, %3;\n\t"                 \
  "add.s64 b1, %2, %6;\n\t"
#define FA_B_STEPS_4 "add.s64 b2, b1, %6;\n\tadd.s64 b3, b2, %6;\n\t"
#define FA_B_STEPS_8 FA_B_STEPS_4 "add.s64 b4, b3, %6;\n\tadd.s64 b5, b4, %6;\n\tadd.s64 b6, b5, %6;\n\tadd.s64 b7, b6, %6;\n\t"
#define FA_MMA_SS(A, B, P) "@e tcgen05.mma.cta_group::1.kind::f16 [%0], " A ", " B ", %3, " P ";\n\t"
#define FA_MMA_TS(A, B, P) "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [" A "], " B ", %3, " P ";\n\t"
#define FA_RUN_ARGS                                                                                   \
  : "r"(d_tmem), "l"(a), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(A_STEP), "n"(B_STEP) : "memory"

template <int NK, uint32_t A_STEP, uint32_t B_STEP>
__device__ __forceinline__ void mma_ss_run_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  static_assert(NK == 2 || NK == 4 || NK == 8, "runs of 2, 4 or 8");
  const uint64_t a = a_desc;
  if constexpr (NK == 2) {
    asm volatile(FA_RUN_HEAD ".reg .b64 a1;\n\tadd.s64 a1, %1, %5;\n\t"
                 FA_MMA_SS("%1", "%2", "p") FA_MMA_SS("a1", "b1", "q") "}" :FA_RUN_ARGS);
  } else if constexpr (NK == 4) {
    asm volatile(FA_RUN_HEAD FA_B_STEPS_4
                 ".reg .b64 a1, a2, a3;\n\tadd.s64 a1, %1, %5;\n\tadd.s64 a2, a1, %5;\n\tadd.s64 a3, a2, %5;\n\t"
                 FA_MMA_SS("%1", "%2", "p") FA_MMA_SS("a1", "b1", "q") FA_MMA_SS("a2", "b2", "q")
                 FA_MMA_SS("a3", "b3", "q") "}" :FA_RUN_ARGS);
  } else {
    asm volatile(FA_RUN_HEAD FA_B_STEPS_8
                 ".reg .b64 a1, a2, a3, a4, a5, a6, a7;\n\t"
                 "add.s64 a1, %1, %5;\n\tadd.s64 a2, a1, %5;\n\tadd.s64 a3, a2, %5;\n\tadd.s64 a4, a3, %5;\n\t"
                 "add.s64 a5, a4, %5;\n\tadd.s64 a6, a5, %5;\n\tadd.s64 a7, a6, %5;\n\t"
                 FA_MMA_SS("%1", "%2", "p") FA_MMA_SS("a1", "b1", "q") FA_MMA_SS("a2", "b2", "q")
                 FA_MMA_SS("a3", "b3", "q") FA_MMA_SS("a4", "b4", "q") FA_MMA_SS("a5", "b5", "q")
                 FA_MMA_SS("a6", "b6", "q") FA_MMA_SS("a7", "b7", "q") "}" :FA_RUN_ARGS);
  }
}

template <int NK, uint32_t A_STEP, uint32_t B_STEP>
__device__ __forceinline__ void mma_ts_run_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  static_assert(NK == 2 || NK == 4 || NK == 8, "runs of 2, 4 or 8");
  const uint32_t a = a_tmem;
#undef FA_RUN_ARGS
#define FA_RUN_ARGS                                                                                   \
  : "r"(d_tmem), "r"(a), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(A_STEP), "n"(B_STEP) : "memory"
  if constexpr (NK == 2) {
    asm volatile(FA_RUN_HEAD ".reg .b32 a1;\n\tadd.u32 a1, %1, %5;\n\t"
                 FA_MMA_TS("%1", "%2", "p") FA_MMA_TS("a1", "b1", "q") "}" :FA_RUN_ARGS);
  } else if constexpr (NK == 4) {
    asm volatile(FA_RUN_HEAD FA_B_STEPS_4
                 ".reg .b32 a1, a2, a3;\n\tadd.u32 a1, %1, %5;\n\tadd.u32 a2, a1, %5;\n\tadd.u32 a3, a2, %5;\n\t"
                 FA_MMA_TS("%1", "%2", "p") FA_MMA_TS("a1", "b1", "q") FA_MMA_TS("a2", "b2", "q")
                 FA_MMA_TS("a3", "b3", "q") "}" :FA_RUN_ARGS);
  } else {
    asm volatile(FA_RUN_HEAD FA_B_STEPS_8
                 ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
                 "add.u32 a1, %1, %5;\n\tadd.u32 a2, a1, %5;\n\tadd.u32 a3, a2, %5;\n\tadd.u32 a4, a3, %5;\n\t"
                 "add.u32 a5, a4, %5;\n\tadd.u32 a6, a5, %5;\n\tadd.u32 a7, a6, %5;\n\t"
                 FA_MMA_TS("%1", "%2", "p") FA_MMA_TS("a1", "b1", "q") FA_MMA_TS("a2", "b2", "q")
                 FA_MMA_TS("a3", "b3", "q") FA_MMA_TS("a4", "b4", "q") FA_MMA_TS("a5", "b5", "q")
                 FA_MMA_TS("a6", "b6", "q") FA_MMA_TS("a7", "b7", "q") "}" :FA_RUN_ARGS);
  }
}
#undef FA_RUN_HEAD
#undef FA_B_STEPS_4
#undef FA_B_STEPS_8
#undef FA_MMA_SS
#undef FA_MMA_TS
#undef FA_RUN_ARGS

// kind::f8f6f4 with A and B in shared memory (K = 32 one-byte elements an
// instruction); the instruction descriptor selects the 8-bit formats.
__device__ __forceinline__ void mma_ss_f8_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 t;\n\telect.sync t|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 t;\n\telect.sync t|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp-collective: thread t reads lane (quarter base + t), 32 consecutive columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Warp-collective: thread t reads lane (quarter base + t), 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Warp-collective: thread t writes lane (quarter base + t), 16 consecutive columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Warp-collective: thread t writes lane (quarter base + t), 32 consecutive columns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ------------------------------------------------------------ descriptors ---
// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), version 1 at bits 46..47, swizzle mode at
// bits 61..63 (2 = 128-byte swizzle).  Operand tiles here are always stored
// in the 128-byte-swizzled layout the TMA unit writes: rows of 128 bytes,
// groups of 8 rows (1024 bytes) as the swizzle atom.
//
//  * K-major (contraction dim contiguous): SBO = 1024 (next 8-row group);
//    LBO unused.  Advance along K inside the 128-byte row by adding bytes.
//  * MN-major (row dim of the product contiguous): LBO = byte distance
//    between 64-element column blocks, SBO = 1024 (next 8 K-rows).
constexpr uint64_t kDescSw128 = (2ull << 61) | (1ull << 46);

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return kDescSw128 | (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, shape
// M x N; a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                  // D format: f32
         | (1u << 7)                // A format: bf16
         | (1u << 10)               // B format: bf16
         | ((uint32_t)a_mn << 15)   // A major-ness
         | ((uint32_t)b_mn << 16)   // B major-ness
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor bit that negates A (kind::f16): the product becomes
// -(A B).  Used for S when the softmax scale is negative, so that everything
// after S works with |scale|.
constexpr uint32_t kIdescNegateA = 1u << 13;

// Instruction descriptor, kind::f8f6f4: E4M3 A and B (format code 0 in both
// type fields), fp32 accumulator, shape M x N, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4)                  // D format: f32
         | (0u << 7) | (0u << 10)   // A, B format: E4M3
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------- numerics ----
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (two lanes of a 64-bit register pair per instruction).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Pack two floats to bf16x2 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void red_add(float* gaddr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(gaddr), "f"(a) : "memory");
}

__device__ __forceinline__ void red_add_v4(float* gaddr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gaddr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

}  // namespace fa
