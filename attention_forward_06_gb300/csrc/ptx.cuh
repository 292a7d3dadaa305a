// ptx.cuh -- hand-written inline-PTX wrappers for sm_103a (Blackwell Ultra):
// mbarriers with bounded waits, TMA tile loads, tcgen05 tensor-memory
// allocation, MMA issue/commit, TMEM loads/stores, and the shared-memory and
// instruction descriptors that tcgen05.mma consumes.  Encodings follow the
// public PTX ISA (tcgen05 "matrix descriptor" and "instruction descriptor"
// tables); the primitive probe kernels check them against CPU matmuls.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace attn {

// ----------------------------------------------------------------------------
// generic helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase has not completed is
// parked by the hardware (for at most `hint_ns`) and woken when it completes,
// so waiting warps do not take issue slots from the warps that share their
// scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// `timeout_ns`.  Returns false on timeout or when *abort becomes non-zero
// (another role gave up); the caller then unwinds without issuing more work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile uint32_t* abort, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// ----------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor): tiled loads into shared memory, completion
// signalled on an mbarrier by transaction bytes.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Converged-warp forms: the whole warp executes the call and one elected lane
// (always the same one, the lowest) performs it.  Keeping the warp converged
// matters: single-lane divergent issue is starved of issue slots when busy warps
// share the scheduler.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_elect(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                                  int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// TMA tile store from shared memory (bulk-group completion), issued by one elected lane.
// Plain (untiled) bulk copy of `bytes` from global to shared memory, completion
// counted on `bar`; both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load_1d_elect(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_store_3d_elect(const CUtensorMap* map, const void* smem_src, int32_t c0,
                                                   int32_t c1, int32_t c2) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];\n\t}" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Close this thread's outstanding bulk stores into a group (only the elected lane has any).
__device__ __forceinline__ void bulk_commit_group_elect() {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.commit_group;\n\t}" ::
          : "memory");
}

// Wait until every bulk store group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every bulk store group of this thread has completed (writes visible).
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Programmatic dependent launch.  griddep_wait: wait until the grids this one depends
// on (the previous kernel of the stream, when launched with programmatic stream
// serialisation) have completed and their memory operations are visible.
// griddep_launch_dependents: let the next such kernel be scheduled once every CTA
// of this grid has signalled or exited.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory (TMEM) and the 5th-generation tensor-core MMA
// ----------------------------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two, 32..512); the whole warp calls
// it; the base address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
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

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T-ish per the descriptors; bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with A read from tensor memory (M rows in lanes, K packed along columns).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, dense tile whose swizzle
// atoms (8 rows x 128 B) start on 1024-byte boundaries:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 49-51  base offset (0: atoms 1024-aligned)
//   bits 61-63  swizzle mode (2 = 128-byte)
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// The same descriptor split in 32-bit halves.  Low word: start address >> 4
// and leading offset >> 4; high word: stride offset >> 4, the fixed 0b001 and
// the swizzle mode.  K steps only move the low word.
__host__ __device__ constexpr uint32_t sdesc_sw128_hi(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}

constexpr uint32_t kNoBar = 0xFFFFFFFFu;

// A whole K loop in one issue: one elected lane issues the MMAs of all K steps
// back to back (the first accumulates into D only if `accumulate`, the rest
// always), then commits them to up to two mbarriers (shared-memory addresses
// bar0, bar1; kNoBar = none: address 0 is a valid shared-memory address).  SS form: A and B descriptors advance by the given
// 16-byte units per step; offsets come from the shared-memory layout.
#define ATTN_COMMITS(B0, B1)                                                                      \
  "setp.ne.b32 c, %" #B0 ", -1;\n\tand.pred c, c, e;\n\t"                                      \
  "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%" #B0 "];\n\t"   \
  "setp.ne.b32 c, %" #B1 ", -1;\n\tand.pred c, c, e;\n\t"                                      \
  "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%" #B1 "];\n\t"
#define ATTN_MMA_SS_STEP(OA, OB)                                      \
  "add.s64 a, %1, " #OA ";\n\tadd.s64 b, %2, " #OB ";\n\t"            \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
__device__ __forceinline__ void mma_bf16_ss_k8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t bar0 = kNoBar, uint32_t bar1 = kNoBar) {
  // K steps of 32 bytes within a 128-byte swizzle atom, then the next 64-column block (16384 B = 1024 units)
  asm volatile(
      "{\n\t.reg .pred e, t, f, c;\n\t.reg .b64 a, b;\n\t"
      "setp.eq.b32 t, 1, 1;\n\tsetp.eq.b32 f, 1, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
      ATTN_MMA_SS_STEP(2, 2) ATTN_MMA_SS_STEP(4, 4) ATTN_MMA_SS_STEP(6, 6)
      ATTN_MMA_SS_STEP(1024, 1024) ATTN_MMA_SS_STEP(1026, 1026) ATTN_MMA_SS_STEP(1028, 1028)
      ATTN_MMA_SS_STEP(1030, 1030) ATTN_COMMITS(4, 5) "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc),
      "r"(bar0), "r"(bar1)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_ss_k4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t bar0 = kNoBar, uint32_t bar1 = kNoBar) {
  asm volatile(
      "{\n\t.reg .pred e, t, f, c;\n\t.reg .b64 a, b;\n\t"
      "setp.eq.b32 t, 1, 1;\n\tsetp.eq.b32 f, 1, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
      ATTN_MMA_SS_STEP(2, 2) ATTN_MMA_SS_STEP(4, 4) ATTN_MMA_SS_STEP(6, 6) ATTN_COMMITS(4, 5) "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(bar0), "r"(bar1)
      : "memory");
}
#undef ATTN_MMA_SS_STEP

// TS form over 8 K steps of 16 keys: A (P in TMEM) advances 8 columns, B (V,
// MN-major) 16 rows of 128 bytes = 128 units per step.
#define ATTN_MMA_TS_STEP(OA, OB)                                      \
  "add.u32 ta, %1, " #OA ";\n\tadd.s64 b, %2, " #OB ";\n\t"           \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, t;\n\t"
__device__ __forceinline__ void mma_bf16_ts_k8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate, uint32_t bar0 = kNoBar, uint32_t bar1 = kNoBar) {
  asm volatile(
      "{\n\t.reg .pred e, t, f, c;\n\t.reg .b64 b;\n\t.reg .b32 ta;\n\t"
      "setp.eq.b32 t, 1, 1;\n\tsetp.ne.b32 f, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, f;\n\t"
      ATTN_MMA_TS_STEP(8, 128) ATTN_MMA_TS_STEP(16, 256) ATTN_MMA_TS_STEP(24, 384) ATTN_MMA_TS_STEP(32, 512)
      ATTN_MMA_TS_STEP(40, 640) ATTN_MMA_TS_STEP(48, 768) ATTN_MMA_TS_STEP(56, 896) ATTN_COMMITS(5, 6) "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(bar0), "r"(bar1)
      : "memory");
}
// TS form over 4 K steps of 16 (K = 64): A advances 8 TMEM columns, B 16 rows per step.
__device__ __forceinline__ void mma_bf16_ts_k4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate, uint32_t bar0 = kNoBar, uint32_t bar1 = kNoBar) {
  asm volatile(
      "{\n\t.reg .pred e, t, f, c;\n\t.reg .b64 b;\n\t.reg .b32 ta;\n\t"
      "setp.eq.b32 t, 1, 1;\n\tsetp.ne.b32 f, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, f;\n\t"
      ATTN_MMA_TS_STEP(8, 128) ATTN_MMA_TS_STEP(16, 256) ATTN_MMA_TS_STEP(24, 384) ATTN_COMMITS(5, 6) "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(bar0), "r"(bar1)
      : "memory");
}
#undef ATTN_MMA_TS_STEP
#undef ATTN_COMMITS

__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Hide a value from the optimiser (stops loop-invariant hoisting of what is derived from it).
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
  asm volatile("" : "+r"(x));
  return x;
}

// Instruction descriptor, kind::f16 with fp16 A/B and fp32 D: the bf16 one with
// both operand formats 0 (f16).  A and B always share one type in a kind::f16 MMA.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D:
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (0 = K), bit 16 B major (0 = K, 1 = MN), bits 17-22 N>>3, bits 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ----------------------------------------------------------------------------
// TMEM <-> registers.  32x32b shape: thread t of the warp reads lane
// (warp's lane quarter)*32 + t, consecutive 32-bit columns.  The load helpers
// include tcgen05.wait::ld in the same asm statement so no use of the
// destination registers can be scheduled before the data has arrived.
// ----------------------------------------------------------------------------
#define ATTN_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                   "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define ATTN_S8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                   "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
      : "r"(taddr)
      : "memory");
}

// One column: this thread's lane of TMEM column `taddr`.
__device__ __forceinline__ uint32_t tmem_ld1_wait(uint32_t taddr) {
  uint32_t v;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v)
      : "r"(taddr)
      : "memory");
  return v;
}

// 128 consecutive columns (four x32 loads issued back to back, one wait).
__device__ __forceinline__ void tmem_ld128_wait(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24), ATTN_R8(32), ATTN_R8(40), ATTN_R8(48),
        ATTN_R8(56), ATTN_R8(64), ATTN_R8(72), ATTN_R8(80), ATTN_R8(88), ATTN_R8(96), ATTN_R8(104),
        ATTN_R8(112), ATTN_R8(120)
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
}

// Two runs of 64 consecutive columns (at a and at b), four x32 loads, one wait.
__device__ __forceinline__ void tmem_ld2x64_wait(uint32_t ta, uint32_t tb, uint32_t (&r)[64], uint32_t (&q)[64]) {
#define ATTN_Q8(b) "=r"(q[b + 0]), "=r"(q[b + 1]), "=r"(q[b + 2]), "=r"(q[b + 3]), \
                   "=r"(q[b + 4]), "=r"(q[b + 5]), "=r"(q[b + 6]), "=r"(q[b + 7])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24), ATTN_R8(32), ATTN_R8(40), ATTN_R8(48), ATTN_R8(56),
        ATTN_Q8(0), ATTN_Q8(8), ATTN_Q8(16), ATTN_Q8(24), ATTN_Q8(32), ATTN_Q8(40), ATTN_Q8(48), ATTN_Q8(56)
      : "r"(ta), "r"(ta + 32), "r"(tb), "r"(tb + 32)
      : "memory");
#undef ATTN_Q8
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      ATTN_S8(0), ATTN_S8(8), ATTN_S8(16), ATTN_S8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef ATTN_R8
#undef ATTN_S8

// ----------------------------------------------------------------------------
// math helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 3-input maximum (one instruction on sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed fp32 pairs in one 64-bit register: element 0 in the low half.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// d = a * b + c on both halves (round to nearest).
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// acc_lo += fp16 in bits 0-15 of `packed`, acc_hi += fp16 in bits 16-31 (mixed-precision adds).
__device__ __forceinline__ void add_f16x2_to_f32(float& acc_lo, float& acc_hi, uint32_t packed) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\t"
      "add.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(packed));
}

// Round two fp32 values to fp16 (nearest-even; beyond 65504 gives infinity) and
// pack: `lo` in bits 0-15, `hi` in 16-31.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// A bf16 pair to the fp16 pair of the same values: exact for magnitudes in
// [2^-14, 65504], rounded to fp16's subnormal grid below, clamped to +-65504 above
// (so a zero weight times an out-of-range value stays zero in a product).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
      : "=r"(d)
      : "f"(__uint_as_float(w & 0xFFFF0000u)), "f"(__uint_as_float(w << 16)));
  return d;
}

// 16-byte shared-memory load and store at a shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Change this warpgroup's per-thread register budget (all four warps execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Round two fp32 values to bf16 (nearest-even) and pack: `lo` in bits 0-15, `hi` in 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

}  // namespace attn
