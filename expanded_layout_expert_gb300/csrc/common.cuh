// Internal device helpers shared by the kernels of libmoe_expand.so:
// status reporting, bounded waits, and inline-PTX wrappers for mbarrier,
// TMA (cp.async.bulk.tensor) and the 5th-generation tensor core (tcgen05).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "moe_expand.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// About two seconds at the GB300's 2.07 GHz maximum SM clock. Every spin in
// this library gives up after this many cycles, records MOE_ERR_TIMEOUT and
// returns, so a broken pipeline cannot hang the GPU.
constexpr long long kWaitLimitCycles = 4000000000LL;

MOE_DEV void set_status(int32_t* st, int code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

MOE_DEV int align_up(int v, int a) { return (v + a - 1) / a * a; }

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

// ---------------------------------------------------------------- mbarrier
MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

MOE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Same test, but a thread whose phase is not complete yet may sleep in it for
// up to `ns` nanoseconds; it wakes as soon as the phase completes. Spinning
// on the plain form returns every few tens of cycles and takes issue slots
// from the other warps of the same scheduler.
MOE_DEV bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Longest sleep of one test inside a bounded wait: short against the wait
// limit, so the abort flag and the limit are still checked often.
constexpr uint32_t kWaitSleepNs = 20000;

// Waits until the phase with the given parity has completed. Gives up when
// *abort becomes non-zero (another role gave up) or after kWaitLimitCycles,
// in which case it records MOE_ERR_TIMEOUT, raises *abort and returns false.
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status,
                       long long limit_cycles = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit_cycles) {
      *abort = 1;
      set_status(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-collective form of mbar_wait: every lane of the warp calls it and all
// lanes leave together, so the loop stays warp-uniform (no per-lane exits to
// reconverge, no separate vote afterwards). Every lane tests the barrier:
// measured on GB300, having lane 0 test it alone and pass the answer on by
// shuffle made the GEMM epilogues 10-18 % slower.
MOE_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status,
                            long long limit_cycles = kWaitLimitCycles) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, kWaitSleepNs))) return true;
    if (__any_sync(0xffffffffu, *abort != 0)) return false;
    if (__any_sync(0xffffffffu, clock64() - t0 > limit_cycles)) {
      *abort = 1;
      set_status(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
MOE_DEV void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled load into shared memory; completion is counted in bytes on `bar`.
// x is the innermost coordinate (bytes for uint8 tensors, a multiple of 16).
MOE_DEV void tma_load_2d(void* dst, const CUtensorMap* tm, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
MOE_DEV void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

MOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05 operation this thread issued
// before has completed.
MOE_DEV void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both operands fp8 (kind::f8f6f4), K = 32.
MOE_DEV void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 TMEM lanes (one per thread of the warp) x 32 consecutive 32-bit
// columns, without waiting: the registers are valid only after a later
// tcgen05.wait::ld (tc_wait64 / tc_regs_landed name them so that no use moves
// above that wait).
MOE_DEV void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// Waits for every TMEM load this thread issued; names two 32-register
// destination arrays so none of their uses can move above the wait.
MOE_DEV void tc_wait64(uint32_t (&v)[32], uint32_t (&w)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]),
                 "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]),
                 "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31]),
                 "+r"(w[0]), "+r"(w[1]), "+r"(w[2]), "+r"(w[3]), "+r"(w[4]), "+r"(w[5]),
                 "+r"(w[6]), "+r"(w[7]), "+r"(w[8]), "+r"(w[9]), "+r"(w[10]), "+r"(w[11]),
                 "+r"(w[12]), "+r"(w[13]), "+r"(w[14]), "+r"(w[15]), "+r"(w[16]),
                 "+r"(w[17]), "+r"(w[18]), "+r"(w[19]), "+r"(w[20]), "+r"(w[21]),
                 "+r"(w[22]), "+r"(w[23]), "+r"(w[24]), "+r"(w[25]), "+r"(w[26]),
                 "+r"(w[27]), "+r"(w[28]), "+r"(w[29]), "+r"(w[30]), "+r"(w[31])
               :
               : "memory");
}

// Register reallocation between warpgroups (all 128 threads of a
// warpgroup execute it).
template <int N>
MOE_DEV void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
MOE_DEV void regs_claim() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms 1024 bytes
// apart (stride byte offset), tile base 1024-byte aligned. Advancing along K
// inside the 128-byte row is done by adding the byte offset to the start
// address; the hardware applies the swizzle to the final address.
MOE_DEV uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address >> 4, bits 0-13
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset, bits 32-45
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                  // swizzle mode: 128-byte
  return d;
}

// Instruction descriptor: dense, D = f32, A = B = e4m3, both K-major.
constexpr uint32_t idesc_f8_f32(int M, int N) {
  return (1u << 4)                                // D format: f32
         | (0u << 7)                              // A format: e4m3
         | (0u << 10)                             // B format: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

// ---- block-scaled MMA (kind::mxf8f6f4): the tensor core applies one ue8m0
// scale per row of A and per row of B to each K = 32 step.

// Generic-proxy writes to shared memory become visible to the async proxy
// (tcgen05.cp, TMA) once this fence has been executed by the writer.
MOE_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory descriptor for a source of 16-byte rows stored back to back
// without swizzling: 8-row core matrices 128 bytes apart (stride byte
// offset); one core matrix wide, so the leading byte offset is unused.
MOE_DEV uint64_t rows16_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address >> 4
  d |= static_cast<uint64_t>(128 >> 4) << 32;           // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (tcgen05)
  return d;                                             // swizzle mode 0: none
}

// Copies 32 rows x 16 bytes from shared memory into TMEM lanes 0-31,
// 4 columns from `taddr`, repeated in all four 32-lane quarters.
MOE_DEV void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D[tmem] (+)= (sfA * A)[smem] * (sfB * B)[smem]^T, e4m3 operands, K = 32,
// one ue8m0 scale per row of A (read from TMEM at sfa) and per row of B
// (at sfb); the byte of each 32-bit scale word is chosen in idesc.
MOE_DEV void tc_mma_mx8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled MMA: D = f32 (implied),
// A = B = e4m3, both K-major, scale factors ue8m0. The scale byte selectors
// (bits 4-5 for B, 29-30 for A) are added per instruction.
constexpr uint32_t idesc_mx8(int M, int N) {
  return (0u << 7)                                // A format: e4m3
         | (0u << 10)                             // B format: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
         | (1u << 23)                             // scale factor type: ue8m0
         | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}
MOE_DEV uint32_t idesc_with_sf(uint32_t idesc, uint32_t a_byte, uint32_t b_byte) {
  return idesc | (b_byte << 4) | (a_byte << 29);
}

// Marks 32 registers as written after a tcgen05.wait::ld that was issued
// earlier, so none of their uses can move above that wait.
MOE_DEV void tc_regs_landed(uint32_t (&v)[32]) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]),
                 "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]),
                 "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// ue8m0 exponent byte -> 2^(byte-127) as fp32 (byte 0 is the subnormal 2^-127).
MOE_DEV float ue8m0_to_f32(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

}  // namespace moe
