// rmsn_tmem.cuh -- tensor memory (TMEM) as per-thread storage for sm_103a kernels.
//
// Each SM has 256 KB of tensor memory: 128 lanes x 512 columns of 32-bit cells.  A CTA
// allocates a power-of-two number of columns (32..512) with tcgen05.alloc; warp w of the
// CTA reaches lanes 32*(w%4) .. 32*(w%4)+31 of every allocated column, its thread with
// lane index i owning lane 32*(w%4)+i.  The 32x32b load/store shapes move, per thread, N
// consecutive columns of its own lane to or from N registers, so a thread can keep an
// array of floats in TMEM and bring one slice at a time into registers.  Warps w, w+4,
// w+8, ... share a lane quadrant and so take disjoint column ranges.
//
// Every tcgen05 instruction here is .sync.aligned: all 32 threads of the warp execute it
// together, converged.  Loads and stores are asynchronous: tcgen05.wait::ld before the
// loaded registers are read, tcgen05.wait::st before a store's cells are loaded again.
// Allocation, its address handed to the other warps through shared memory, and the
// release follow the tcgen05 fence rules: fence::before_thread_sync before the thread
// barrier that publishes (or retires) TMEM state, fence::after_thread_sync after it.
#pragma once

#include <stdint.h>

namespace rmsn {

// Columns a CTA allocates: the least power of two >= n, at least 32 (n <= 512).
__host__ __device__ constexpr uint32_t tmem_alloc_cols(uint32_t n) {
  uint32_t c = 32;
  while (c < n) c <<= 1;
  return c;
}

// One whole warp: allocates `ncols` columns and writes their base address to *dst
// (shared memory), then gives up the CTA's right to allocate again.
__device__ __forceinline__ void tmem_alloc_warp(uint32_t* dst, uint32_t ncols) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(a),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// One whole warp (the one that allocated): releases the columns.
__device__ __forceinline__ void tmem_dealloc_warp(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The address of column `col` in this warp's lane quadrant.
__device__ __forceinline__ uint32_t tmem_warp_addr(uint32_t base, uint32_t warp, uint32_t col) {
  return base + ((32u * (warp & 3u)) << 16) + col;
}

// 16 consecutive columns of this thread's lane <-> r[0..15].
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]),
        "=f"(r[7]), "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]),
        "=f"(r[13]), "=f"(r[14]), "=f"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]),
      "f"(r[8]), "f"(r[9]), "f"(r[10]), "f"(r[11]), "f"(r[12]), "f"(r[13]), "f"(r[14]),
      "f"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace rmsn
