// Thin inline-PTX wrappers for the Blackwell (sm_103a) features the attention
// kernels use: mbarriers, TMA bulk-tensor copies, tcgen05 MMA into tensor memory
// (TMEM), TMEM loads/stores and the fences that order them.  Every wait is
// bounded: it gives up after a deadline, records an error code in a device status
// word and returns false, so no kernel can spin forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace fa {

// Error codes written to the device status word (match fa_status in fa_gb300.h).
constexpr unsigned kErrTimeout = 4u;

// Give up on a wait after this many nanoseconds of %globaltimer (1 s).  The failure-
// path test build compiles with a few milliseconds instead (FA_WAIT_LIMIT_NS).
#ifndef FA_WAIT_LIMIT_NS
#define FA_WAIT_LIMIT_NS (1000ull * 1000ull * 1000ull)
#endif
constexpr unsigned long long kWaitLimitNs = FA_WAIT_LIMIT_NS;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Shared per-CTA abort flag plus the device status word.  Once any wait in the CTA
// times out, later waits return false at once so every role drains quickly.
struct WaitCtx {
  volatile int* abort_flag;     // shared memory
  unsigned int* status;         // global memory (may be null)
};

// Wait until the phase with the given parity of `bar` has completed.
// Returns false (after recording kErrTimeout) if the deadline passes or the CTA
// is already aborting.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long start = globaltimer();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0u) {
      if (*w.abort_flag) return false;
      if (globaltimer() - start > kWaitLimitNs) {
        *w.abort_flag = 1;
        if (w.status) atomicCAS(w.status, 0u, kErrTimeout);
        return false;
      }
    }
  }
}

// Bounded wait used while draining after an abort: never sets new errors.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  unsigned long long start = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - start > limit_ns) return;
  }
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(smem_src))
               : "memory");
}

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Programmatic dependent launch.  launch_dependents lets the next kernel of the stream
// (launched with programmatic stream serialization) start launching its CTAs once every
// CTA of this grid has executed it; griddep_wait blocks until the kernels this grid
// depends on have completed and their memory operations are visible.  A kernel launched
// without the attribute returns from griddep_wait at once.
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Wait until every bulk copy this thread committed has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the async proxy
// (TMA engine and tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `nthreads` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
//   start: shared address of the first element (16-byte units in bits 0-13)
//   lbo:   leading-dimension byte offset (bits 16-29)
//   sbo:   stride-dimension byte offset (bits 32-45)
//   bits 46-47 = 1 (descriptor version), bits 61-63 = 2 (128-byte swizzle).
// The tile must sit on a 1024-byte boundary; offsets inside a swizzle atom are
// expressed by moving `start`, because the swizzle is a function of address bits.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t start, uint32_t lbo, uint32_t sbo) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  desc |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  desc |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  desc |= static_cast<uint64_t>(1u) << 46;
  desc |= static_cast<uint64_t>(2u) << 61;
  return desc;
}

// The same descriptor moved by `bytes` (a multiple of 16): only the start-address
// field changes, and it cannot carry out of its 14 bits for addresses inside the
// 228 KB shared window, so a plain add replaces re-encoding the descriptor.
__device__ __forceinline__ uint64_t sdesc_adv(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// Instruction descriptor, kind::f16 with bf16 A and B and an fp32 accumulator.
//   bits 4-5 D format (1 = f32); 7-9 A format (1 = bf16); 10-12 B format (1 = bf16);
//   bit 15 A major (0 = K-major, 1 = M-major); bit 16 B major (0 = K-major, 1 = N-major);
//   bits 17-22 N >> 3; bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]; one thread issues.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; one thread issues.  A (M = 128 rows = lanes) holds
// two bf16 K-elements per 32-bit column: column c of a lane = (element 2c in the low
// half, element 2c+1 in the high half), so each K = 16 step advances 8 columns.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f8f6f4 with A and B both E4M3 (format code 0 in
// bits 7-9 and 10-12), fp32 accumulator, both operands K-major.  One MMA consumes
// K = 32 elements: 32 bytes of each operand row, the same byte step as bf16's K = 16.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Eight kind::f16 MMAs from shared memory into one accumulator, one K = 16 step each:
// descriptor k of A (B) is `a` (`b`) plus the compile-time offset Ak (Bk), in the
// descriptor's 16-byte units.  The first MMA accumulates when `acc` is non-zero, the
// other seven always.  One asm block: the predicates are set once and each step is two
// adds and the MMA, which keeps the single issuing thread ahead of the tensor pipe.
template <uint32_t A0, uint32_t A1, uint32_t A2, uint32_t A3, uint32_t A4, uint32_t A5, uint32_t A6, uint32_t A7,
          uint32_t B0, uint32_t B1, uint32_t B2, uint32_t B3, uint32_t B4, uint32_t B5, uint32_t B6, uint32_t B7>
__device__ __forceinline__ void mma8_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
      "add.s64 da, %1, %6;\n\tadd.s64 db, %2, %14;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p0;\n\t"
      "add.s64 da, %1, %7;\n\tadd.s64 db, %2, %15;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %8;\n\tadd.s64 db, %2, %16;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %9;\n\tadd.s64 db, %2, %17;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %10;\n\tadd.s64 db, %2, %18;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %11;\n\tadd.s64 db, %2, %19;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %12;\n\tadd.s64 db, %2, %20;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %13;\n\tadd.s64 db, %2, %21;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p1;\n\t}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(1u),
      "n"(A0), "n"(A1), "n"(A2), "n"(A3), "n"(A4), "n"(A5), "n"(A6), "n"(A7),
      "n"(B0), "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6), "n"(B7)
      : "memory");
}

// The same with A from tensor memory (the TS form): step k reads A at a_tmem + 8k
// (two bf16 K-elements per 32-bit column, so K = 16 is eight columns) and B at b plus
// the k-th offset.
template <uint32_t B0, uint32_t B1, uint32_t B2, uint32_t B3, uint32_t B4, uint32_t B5, uint32_t B6, uint32_t B7>
__device__ __forceinline__ void mma8_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 db;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
      "add.s64 db, %2, %6;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p0;\n\t"
      "add.u32 ta, %1, 8;\n\tadd.s64 db, %2, %7;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, %1, 16;\n\tadd.s64 db, %2, %8;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, %1, 24;\n\tadd.s64 db, %2, %9;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, %1, 32;\n\tadd.s64 db, %2, %10;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, %1, 40;\n\tadd.s64 db, %2, %11;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, %1, 48;\n\tadd.s64 db, %2, %12;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t"
      "add.u32 ta, %1, 56;\n\tadd.s64 db, %2, %13;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, p1;\n\t}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(1u),
      "n"(B0), "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6), "n"(B7)
      : "memory");
}

// Four kind::f8f6f4 MMAs (E4M3 A and B from shared memory, K = 32 each) into one
// accumulator, offsets as in mma8_bf16_ss.
template <uint32_t A0, uint32_t A1, uint32_t A2, uint32_t A3, uint32_t B0, uint32_t B1, uint32_t B2, uint32_t B3>
__device__ __forceinline__ void mma4_f8_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
      "add.s64 da, %1, %6;\n\tadd.s64 db, %2, %10;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, p0;\n\t"
      "add.s64 da, %1, %7;\n\tadd.s64 db, %2, %11;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %8;\n\tadd.s64 db, %2, %12;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, p1;\n\t"
      "add.s64 da, %1, %9;\n\tadd.s64 db, %2, %13;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, p1;\n\t}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(1u),
      "n"(A0), "n"(A1), "n"(A2), "n"(A3), "n"(B0), "n"(B1), "n"(B2), "n"(B3)
      : "memory");
}

// Two kind::f8f6f4 MMAs with A from tensor memory (four E4M3 K-elements per column, so
// K = 32 is eight columns): step k reads A at a_tmem + 8k and B at b plus the k-th offset.
template <uint32_t B0, uint32_t B1>
__device__ __forceinline__ void mma2_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 db;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
      "add.s64 db, %2, %6;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], db, %3, p0;\n\t"
      "add.u32 ta, %1, 8;\n\tadd.s64 db, %2, %7;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], db, %3, p1;\n\t}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(1u), "n"(B0), "n"(B1)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// TMEM -> registers: the calling warp reads 32 lanes (its quarter) x 32 columns of
// 32-bit values; thread t gets lane (base lane + t).  The wait is folded into the
// same asm statement so no use of the registers can be scheduled before it.
#define FA_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}
#undef FA_R8

// TMEM -> registers, 32 lanes x 64 columns in one load and one wait (half the
// exposed load latency of two 32-column loads).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// Registers -> TMEM, same 32 lanes x 32 columns shape; waits for completion.
#define FA_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}
#undef FA_W8

// TMEM -> registers, 32 lanes x 128 columns in one load and one wait (a whole score
// row per thread at one load latency).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// Registers -> TMEM, 32 lanes x 64 columns in one store and one wait.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}

// ------------------------------------------------------------ small numerics

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Paired fp32 ops on two lanes at once (f32x2): (d0, d1) = (a0, a1) * b + c.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\tmov.b64 z, {%5, %5};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (s0, s1) += (a0, a1)
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 x, y, z;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// (d0, d1) = (a0 - c, a1 - c) * (b0, b1)
__device__ __forceinline__ void fsubmul2(float& d0, float& d1, float a0, float a1, float c, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\tmov.b64 z, {%5, %6};\n\t"
      "sub.rn.f32x2 w, x, y;\n\tmul.rn.f32x2 w, w, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(c), "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four floats -> four E4M3 values (round to nearest even, saturating at +-448) in one
// word, x0 in the lowest byte.  cvt puts its first source in the upper byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// 16 bytes from shared memory (the counterpart of st_shared_v4).
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// A global load that stays where it is written (the compiler may otherwise sink a
// prefetch down to its first use and expose the whole memory latency there).
__device__ __forceinline__ float ld_global_pinned(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_global_pinned(const int* p) {
  int v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a 128-byte-swizzled
// tile whose rows are 128 bytes apart (the layout TMA writes for SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// The same for SWIZZLE_64B with 64-byte rows: address bits 4-5 (the chunk, 0..3) are
// XOR-ed with address bits 7-8, i.e. with (row / 2) mod 4.
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk) {
  return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

}  // namespace fa
