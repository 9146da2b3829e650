// umma.cuh -- the tcgen05 (fifth-generation tensor core) operations used by
// the GQA score kernel, as inline PTX for sm_103a: tensor-memory allocation,
// the shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle, the instruction descriptor of a kind::f16 MMA with fp32
// accumulation, the MMA itself, its completion signal on an mbarrier, and the
// load of accumulator rows back into registers.
//
// Operand layout (K-major, 128-byte swizzle): each row of the operand holds
// 64 fp16 elements of K in 128 bytes; 8 consecutive rows form a 1024-byte
// atom whose 16-byte chunks are permuted by chunk ^= (row % 8); atoms follow
// each other along M (or N) every 1024 bytes, and the next 64 elements of K
// start a new column of atoms. An MMA consumes K = 16 (32 bytes of a row), so
// successive MMAs advance the descriptor's start address by 32 bytes inside
// an atom and by a whole atom column every four MMAs.
#pragma once

#include <cuda_runtime.h>

#include <stdint.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

// Byte offset of the 8-byte piece at byte b (b % 8 == 0) of row r inside one
// 64-element column of a 128-byte-swizzled K-major operand.
__device__ __forceinline__ uint32_t sw128_offset(int r, int b) {
  return static_cast<uint32_t>(r * 128 + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15)));
}

// Shared-memory matrix descriptor: start address (bits 0-13, >> 4), leading
// byte offset (16-29; unused by a swizzled K-major operand whose MMA K fits
// in one 128-byte row), stride byte offset between 8-row atoms (32-45),
// descriptor version 1 (46-47), base offset 0 (atoms are 1024-byte aligned),
// swizzle mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
constexpr uint32_t f16_idesc(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// One warp allocates ncols tensor-memory columns (a power of two >= 32) and
// writes their base address to *slot; the permit is given up right away so
// that other CTAs on the SM can allocate.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Bounded wait for phase `parity` of an mbarrier that suspends the thread
// (up to ~1 us per try, woken when the phase completes) instead of spinning,
// so that waiting warps leave the issue slots to the working ones; gives up
// after ~2 s like mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
        : "memory");
    if (ok) return true;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}

// One lane of the (converged) warp is elected: true there, false elsewhere.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(pred));
  return pred != 0;
}

// Bounded wait that backs off with growing sleeps (32 ns doubling to 512
// ns) between tries, for waits that are expected to be long: a sleeping
// warp issues nothing.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (mbar_try_wait(bar, parity)) return true;
    ns = ns < 512 ? 2 * ns : ns;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}

// Plain arrival on an mbarrier (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Ordering of tensor-core operations around thread synchronisation.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// Arrive (once) on the mbarrier when every MMA issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Eight consecutive 32-bit columns of one tensor-memory lane per thread:
// thread t of the warp reads lane (taddr.lane + t). A warp may only address
// its own quarter of the lanes (32 * (warp % 4) ...).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace
}  // namespace tri
