// rmsn_common.cuh -- device helpers shared by the forward and backward kernels.
//
// Staging model (both kernels): a CTA owns a contiguous chunk of normalized rows.  One
// producer thread streams the chunk's rows from HBM into an S-stage shared-memory ring
// with 1-D bulk asynchronous copies (cp.async.bulk, the TMA engine's untiled form), each
// stage guarded by a "full" mbarrier (transaction bytes) and an "empty" mbarrier
// (consumer releases).  Consumers are G row groups of NTg threads; group g takes row slot
// g of every stage, and each thread owns the same VPT 16-byte column vectors of every row
// it touches (column vector c = lt + v*NTg), so per-column state (the weight, the dw
// partial sums) lives in registers for the whole chunk.  The producer has a warp of its
// own: issuing a stage's copies takes long enough that, done by a consumer warp, it would
// sit on the slowest warp's path every stage.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

// Device-side error bits (see rmsnorm_train_device_error in the public header).
enum : unsigned { kErrConsumerWait = 1u, kErrProducerWait = 2u };

// A bounded wait gives up after this many nanoseconds of %globaltimer spent waiting.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
// Waiting time is summed poll by poll; a step between two polls that goes backwards or
// is longer than this is the timer being set (or the context being off the GPU), not
// time spent waiting, and is not counted.  Without this, one backward step of the timer
// would read as a wait of ~2^64 ns and abort a healthy kernel.
constexpr unsigned long long kWaitStepMaxNs = 1000000ull;  // 1 ms


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Adds the time since the previous poll (`prev`, then updated) to `waited`, skipping
// steps the timer took outside the wait; true once `waited` passes the limit.
__device__ __forceinline__ bool wait_expired(unsigned long long& prev,
                                             unsigned long long& waited) {
  const unsigned long long now = global_ns();
  const unsigned long long step = now - prev;  // huge if the timer stepped back
  prev = now;
  if (step <= kWaitStepMaxNs) waited += step;
  return waited > kWaitLimitNs;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One attempt to wait for phase `parity` of `bar` (the hardware may suspend the thread
// for a while before answering "not yet").
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete.  Bounded: after kWaitLimitNs it records
// `errbit` in the device error word, raises the CTA's abort flag and returns false.  Once
// the abort flag is up every later wait returns at once, so all threads still run the
// same barriers (no named barrier can then hang) and the CTA drains and exits.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag,
                                                  unsigned* err_word, unsigned errbit) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long prev = global_ns(), waited = 0;
  for (;;) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (wait_expired(prev, waited)) {
      atomicOr(err_word, errbit);
      *abort_flag = 1;
      return false;
    }
  }
}

// The producer's last step: waits until the `issued` stages' copies have landed (the last
// S of them; earlier ones were released by the consumers), so that no copy still writes
// this CTA's shared memory once it exits -- also after an abort, whose flag it ignores.
// Bounded by one kWaitLimitNs for the whole drain.
__device__ __forceinline__ void mbar_drain(uint64_t* full, int S, int32_t issued) {
  unsigned long long prev = global_ns(), waited = 0;
  for (int32_t j = issued > S ? issued - S : 0; j < issued; ++j) {
    const uint32_t parity = static_cast<uint32_t>(j / S) & 1u;
    while (!mbar_try_wait(&full[j % S], parity))
      if (wait_expired(prev, waited)) return;
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// A row kernel's barriers, initialised by the 32 lanes of one warp (a barrier a lane, each
// lane fencing its own inits): the ring's S full barriers (one arrival: the producer's
// expect-tx), its S empty barriers (`empty_count` arrivals) and `nred` per-row reduction
// barriers (`red_count` arrivals).  One thread doing them all in series costs ~7 ns a
// barrier, which the kernel's start waits on.  The caller's __syncthreads() publishes them.
__device__ __forceinline__ void init_row_barriers_warp(uint64_t* full, uint64_t* empty, int S,
                                                       uint32_t empty_count, uint64_t* redb,
                                                       int nred, uint32_t red_count,
                                                       int lane) {
  for (int i = lane; i < 2 * S + nred; i += 32) {
    if (i < S)
      mbar_init(&full[i], 1u);
    else if (i < 2 * S)
      mbar_init(&empty[i - S], empty_count);
    else
      mbar_init(&redb[i - 2 * S], red_count);
  }
  fence_barrier_init();
}

// L2 policy for data that is read exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared, completing `bytes` transaction bytes on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// Makes `bar` track this thread's earlier cp.async copies: adds one pending arrival to
// the current phase now and performs that arrival once the copies have landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's memory, and allow the next
// grid to be scheduled early.  Both are no-ops when the launch did not opt in.
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- packed FP32 pairs (sm_100+ f32x2 arithmetic, one instruction for two lanes) -----
//
// A pair lives in one 64-bit register pair; every operation rounds each lane to nearest
// even exactly as its scalar counterpart would (no flush to zero).

struct f2 {
  unsigned long long v;
};

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f2 f2_splat(float a) { return f2_make(a, a); }
__device__ __forceinline__ float f2_lo(f2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
  return lo;
}
__device__ __forceinline__ float f2_hi(f2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
  return hi;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
// a * b + c with one rounding per lane
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// One word of two BF16 (low half = element 2i) -> the pair of their FP32 values (exact).
__device__ __forceinline__ f2 bf2_to_f2(uint32_t u) {
  return f2_make(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
// The two elementwise products of two words of two BF16 each, as an FP32 pair: exact (a
// product of two 8-bit significands fits FP32's 24), formed by the mixed-precision fma
// (BF16 sources, FP32 accumulator) with no conversion of either word.
__device__ __forceinline__ f2 bf2_mul_exact(uint32_t a, uint32_t b) {
  f2 r;
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t.reg .f32 p0, p1;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.bf16 p0, a0, b0, 0f80000000;\n\t"
      "fma.rn.f32.bf16 p1, a1, b1, 0f80000000;\n\t"
      "mov.b64 %0, {p0, p1};\n\t}"
      : "=l"(r.v)
      : "r"(a), "r"(b));
  return r;
}
// c + a*a per lane for the two BF16 of word a (one rounding each: the square is exact).
__device__ __forceinline__ f2 bf2_sq_acc(uint32_t a, f2 c) {
  f2 r;
  asm("{\n\t.reg .b16 a0, a1;\n\t.reg .f32 c0, c1, p0, p1;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b64 {c0, c1}, %2;\n\t"
      "fma.rn.f32.bf16 p0, a0, a0, c0;\n\t"
      "fma.rn.f32.bf16 p1, a1, a1, c1;\n\t"
      "mov.b64 %0, {p0, p1};\n\t}"
      : "=l"(r.v)
      : "r"(a), "l"(c.v));
  return r;
}

// The pair rounded to two BF16 (nearest even), element 2i in the low half.
__device__ __forceinline__ uint32_t f2_to_bf2(f2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- BF16 packing --------------------------------------------------------------------

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two FP32 values -> one word of two BF16 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// 16 bytes of shared memory at the shared-window address a (32-bit addressing).
__device__ __forceinline__ uint4 lds128_at(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f_at(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ void stg128(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x);
  f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z);
  f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  u.x = pack_bf2(f[0], f[1]);
  u.y = pack_bf2(f[2], f[3]);
  u.z = pack_bf2(f[4], f[5]);
  u.w = pack_bf2(f[6], f[7]);
  return u;
}

// Loads the 8 weights of column vector c as FP32.
template <bool kFp32W>
__device__ __forceinline__ void load_w8(const void* w, int c, float (&f)[8]) {
  if constexpr (kFp32W) {
    const float4* p = reinterpret_cast<const float4*>(w) + 2 * c;
    float4 a = __ldg(p), b = __ldg(p + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(w) + c);
    unpack8(u, f);
  }
}

// Loads the 8 weights of column vector c as four FP32 pairs.
template <bool kFp32W>
__device__ __forceinline__ void load_w8_pairs(const void* w, int c, f2 (&p)[4]) {
  if constexpr (kFp32W) {
    const float4* q = reinterpret_cast<const float4*>(w) + 2 * c;
    float4 a = __ldg(q), b = __ldg(q + 1);
    p[0] = f2_make(a.x, a.y);
    p[1] = f2_make(a.z, a.w);
    p[2] = f2_make(b.x, b.y);
    p[3] = f2_make(b.z, b.w);
  } else {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(w) + c);
    p[0] = bf2_to_f2(u.x);
    p[1] = bf2_to_f2(u.y);
    p[2] = bf2_to_f2(u.z);
    p[3] = bf2_to_f2(u.w);
  }
}

__device__ __forceinline__ uint32_t u4_get(const uint4& u, int q) {
  return q == 0 ? u.x : (q == 1 ? u.y : (q == 2 ? u.z : u.w));
}

// Butterfly sum over a warp: every lane ends with the same bits (a+b == b+a exactly).
__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over an aligned group of `ntg` lanes (ntg = 8 or 16) by butterfly; every lane of
// the group gets the same bits.
__device__ __forceinline__ float subwarp_allsum(float v, int ntg) {
  for (int o = ntg >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of a row's nw per-warp partials in slot order (nw <= 16; the slot row is 16-byte
// aligned, so four vector loads cover it).  Every thread gets the same bits.
__device__ __forceinline__ float slot_sum(const float* slot, int nw) {
  float acc = 0.f;
  for (int i = 0; i < nw; i += 4) {
    const float4 q = *reinterpret_cast<const float4*>(slot + i);
    acc += q.x;
    if (i + 1 < nw) acc += q.y;
    if (i + 2 < nw) acc += q.z;
    if (i + 3 < nw) acc += q.w;
  }
  return acc;
}

// ---- row addressing and the producer -------------------------------------------------

// Row r = (token t, head h) = (r / nh, r % nh) starts at element t*s_tok + h*s_head.
struct RowMap {
  int32_t nh;
  int32_t H;
  int64_t s_tok;
  int64_t s_head;
};

// Copies rows [ra, rb) of a BF16 tensor into consecutive H-element slots at `dst`.  When
// a token's heads are back to back (s_head == H) the rows of one token form one run and
// take one bulk copy, so the walk costs one step per token touched, not per row (the
// producer's time between a slot's release and the slot's copies adds to every stage's
// turnaround).  Otherwise every row is its own copy.  One division per call.
__device__ __forceinline__ void copy_rows(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                          const RowMap& m, int32_t ra, int32_t rb,
                                          uint64_t* bar, uint64_t pol) {
  int32_t t = ra / m.nh;
  int32_t h = ra - t * m.nh;
  const uint32_t row_bytes = static_cast<uint32_t>(m.H) * 2u;
  __nv_bfloat16* d = dst;
  if (m.s_head == m.H) {
    for (int32_t r = ra; r < rb; ++t, h = 0) {
      const int32_t n = min(rb - r, m.nh - h);
      bulk_g2s(d, src + static_cast<int64_t>(t) * m.s_tok + static_cast<int64_t>(h) * m.H,
               static_cast<uint32_t>(n) * row_bytes, bar, pol);
      d += static_cast<int64_t>(n) * m.H;
      r += n;
    }
  } else {
    int64_t off = static_cast<int64_t>(t) * m.s_tok + static_cast<int64_t>(h) * m.s_head;
    for (int32_t r = ra; r < rb; ++r, d += m.H) {
      bulk_g2s(d, src + off, row_bytes, bar, pol);
      if (++h == m.nh) {
        h = 0;
        ++t;
        off = static_cast<int64_t>(t) * m.s_tok;
      } else {
        off += m.s_head;
      }
    }
  }
}

// Contiguous [R, H] tensor: rows [ra, rb) in one copy.
__device__ __forceinline__ void copy_rows_contig(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                                 int32_t H, int32_t ra, int32_t rb,
                                                 uint64_t* bar, uint64_t pol) {
  bulk_g2s(dst, src + static_cast<int64_t>(ra) * H,
           static_cast<uint32_t>(rb - ra) * static_cast<uint32_t>(H) * 2u, bar, pol);
}

// ---- host helpers of every kernel translation unit (defined in rmsn_api.cu) ----
// Opts fn into the shared-memory size the row kernels use (once per device).
cudaError_t prepare_kernel(const void* fn, size_t smem);
// Resident CTAs an SM of fn at this block size and shared memory (cached per device).
int blocks_per_sm(const void* fn, int threads, size_t smem);
// Launches fn with programmatic dependent launch (its prologue may overlap the previous
// kernel on the stream).
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       void** args);

}  // namespace rmsn
