// ln_common.cuh -- device helpers of the LayerNorm kernels beyond rmsn_common.cuh: the
// thread-block-cluster operations of the CTA-pair builds (hidden sizes above 8192, where
// one row's columns are split between the two CTAs of a cluster, on two SMs).
//
// A pair exchanges each row's per-warp partial sums through distributed shared memory: a
// warp stores its partial into the peer CTA's reduction slots (st.shared::cluster) and
// arrives on the peer's reduction barrier with release semantics at cluster scope; the
// peer's waiters acquire at cluster scope.  Every remote access happens between two
// cluster barriers: one after the barriers are initialised, one before either CTA exits.
#pragma once

#include "rmsn_common.cuh"
#include "rmsn_tmem.cuh"

namespace lnorm {

using namespace rmsn;

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the variable at `p` (this CTA's shared memory) in the
// CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}

__device__ __forceinline__ void st_peer_f2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_peer(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait_bounded with acquire at cluster scope: the barrier's arrivals include the peer
// CTA's, which release its stores into this CTA's shared memory.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t* bar, uint32_t parity,
                                                          volatile int* abort_flag,
                                                          unsigned* err_word, unsigned errbit) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  unsigned long long prev = global_ns(), waited = 0;
  for (;;) {
    if (*abort_flag) return false;
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (wait_expired(prev, waited)) {
      atomicOr(err_word, errbit);
      *abort_flag = 1;
      return false;
    }
  }
}

// All threads of both CTAs of the cluster; every thread of a warp executes it together.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Rows [ra, rb) of a row-major [R, H] BF16 tensor, columns [col0, col0 + Hc), into
// consecutive Hc-element slots at `dst`: one bulk copy per row (the half-rows are not
// contiguous).  Hc * 2 and col0 * 2 are multiples of 16 bytes.
__device__ __forceinline__ void copy_half_rows(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                               int32_t H, int32_t Hc, int32_t col0, int32_t ra,
                                               int32_t rb, uint64_t* bar, uint64_t pol) {
  const uint32_t bytes = static_cast<uint32_t>(Hc) * 2u;
  for (int32_t r = ra; r < rb; ++r, dst += Hc)
    bulk_g2s(dst, src + static_cast<int64_t>(r) * H + col0, bytes, bar, pol);
}

// The 8 weights (or biases) of one column vector, kept in registers as loaded: BF16 as one
// uint4 of pairs (half the registers of FP32), FP32 as two float4.
template <bool kFp32>
struct Param8;
template <>
struct Param8<false> {
  uint4 u;
};
template <>
struct Param8<true> {
  float4 a, b;
};

// Loads column vector c (elements 8c .. 8c+7) of a BF16 or FP32 parameter array.
template <bool kFp32>
__device__ __forceinline__ void load_param8(const void* p, int c, Param8<kFp32>& out) {
  if constexpr (kFp32) {
    const float4* q = reinterpret_cast<const float4*>(p) + 2 * c;
    out.a = __ldg(q);
    out.b = __ldg(q + 1);
  } else {
    out.u = __ldg(reinterpret_cast<const uint4*>(p) + c);
  }
}

// x - k for the two BF16 of word u, as an FP32 pair, each rounded once (the same bits as
// converting x and subtracting in FP32): the mixed-precision fma x*1 + (-k), which reads
// the BF16 halves of the word with no conversion.  nk = -k.
__device__ __forceinline__ f2 bf2_minus(uint32_t u, float nk) {
  f2 r;
  asm("{\n\t.reg .b16 a0, a1, one;\n\t.reg .f32 p0, p1;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b16 one, 0x3F80;\n\t"
      "fma.rn.f32.bf16 p0, a0, one, %2;\n\t"
      "fma.rn.f32.bf16 p1, a1, one, %2;\n\t"
      "mov.b64 %0, {p0, p1};\n\t}"
      : "=l"(r.v)
      : "r"(u), "f"(nk));
  return r;
}

// Elements 2q and 2q+1 of a column vector's parameters, as an FP32 pair (q a constant
// after unrolling).
template <bool kFp32>
__device__ __forceinline__ f2 param_pair(const Param8<kFp32>& p, int q) {
  if constexpr (kFp32) {
    return q == 0 ? f2_make(p.a.x, p.a.y)
                  : (q == 1 ? f2_make(p.a.z, p.a.w)
                            : (q == 2 ? f2_make(p.b.x, p.b.y) : f2_make(p.b.z, p.b.w)));
  } else {
    return bf2_to_f2(u4_get(p.u, q));
  }
}

// 8 consecutive tensor-memory columns of this thread's lane <-> r[0..7] (the 32x32b
// shape, as rmsn_tmem.cuh's 16-column forms; whole warp, .sync.aligned).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]),
                 "=f"(r[6]), "=f"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"r"(taddr), "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]),
               "f"(r[6]), "f"(r[7])
               : "memory");
}

}  // namespace lnorm
