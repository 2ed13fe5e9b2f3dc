// rmsn_bwd_rows.cuh -- the RMSNorm training backward's row pass for sm_103a: dx fused with
// the compensated dw partial sums, one program for both modes (the partition is chosen at
// run time: a fixed chunk of rows per CTA, or a fixed prefix plus rows handed out from a
// counter).  Included by rmsn_bwd.cu (builds that read rstd) and rmsn_bwd_rc.cu (builds
// that recompute it); each CTA writes one dw partial to the workspace, and the fixed-order
// finish kernel (rmsn_bwd.cu) adds them.
//
// Per normalized row, with r the forward's rstd (flashinfer PR #8827, description: the
// backward's BF16 dx and FP32 dw; the residual form's combined gradient):
//   xhat_j = x_j * r,  g_j = dy_j * w_j,  c = (1/H) sum_j g_j * xhat_j
//        = (r/H) * sum_j (dy_j * w_j) * x_j
//   dx_j   = BF16((g_j - xhat_j * c) * r  [+ dh_j])
//   dw_j  += dy_j * xhat_j          over every row of every CTA's rows
//
// dw accuracy (PR #8849 and PR #8827's route notes: every dw element within
// atol 1e-4 + rtol 1e-4 of an FP64 sum, a budget plain FP32 running sums break at large
// T).  Two error sources are removed: the rounding of each product and the rounding of
// each addition.  With rstd split as rs_hi (its top 8 significant bits) + rs_lo, the
// product dy*x*rs_hi is exact in FP32 (dy*x carries at most 16 significant bits), and
// dy*x*rs_lo is 2^-8 smaller.  Each consumer thread keeps per column a running FP32 sum
// of the exact products and a compensation term that collects each addition's Fast2Sum
// error plus the small dy*x*rs_lo terms.  A CTA's groups combine into an unevaluated
// (hi, lo) FP32 pair per column, written as the CTA's partial; the finish kernel adds the
// P pairs in a fixed order with Knuth's TwoSum, so dw is bit-reproducible whenever the
// row -> CTA mapping is (deterministic builds: fixed by (R, P)).  What remains is about the
// final rounding of dw to FP32.  dx never depends on the partition: it is bit-identical
// across modes.
//
// Split-phase rows (see the consumer loop) keep the row reduction off the critical path.
// Arithmetic runs on packed FP32 pairs (f32x2): two columns per instruction.
#pragma once

#include "rmsn_common.cuh"
#include "rmsn_launch.h"
#include "rmsn_tmem.cuh"

namespace rmsn {

// Knuth's TwoSum: s + err == a + b exactly, no ordering assumption.
__device__ __forceinline__ float two_sum(float a, float b, float& err) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bp);
  err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
  return s;
}

// The non-deterministic row counter's two words: ctl[0] the tag of the call that opened
// the pool of tail rows (a nonzero per-call number), ctl[1] the next tail row.
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// First row of CTA k's chunk in the deterministic partition of R rows over P CTAs.
__device__ __forceinline__ int32_t r0_det(int32_t k, int32_t R, int32_t P) {
  return static_cast<int32_t>((static_cast<int64_t>(k) * R) / P);
}

// A row's two reduced sums: (dy*w)*x, and x^2 (builds that recompute rstd).
struct RowSums {
  float dot, ss;
};

// Launch bounds per shape class (rmsn_launch.h): narrow CTAs of up to 256 consumers, two
// an SM; multi-group CTAs of up to 480 consumers and wide CTAs (384 consumers with
// 2-vector threads, 256 with 4-vector threads), one an SM; each + the producer warp.
//
// kRc = true: the backward is not handed rstd; phase A forms sum_j x_j^2 beside
// sum_j (dy_j*w_j)*x_j (both through the one reduction) and phase B recomputes
// rstd = 1/sqrt(sum x^2 / H + eps) as the forward does, writing it to a.rstd_out if given.
// The rows a CTA takes (the producer decides them stage by stage and passes each stage's
// rows [start, end) to the consumers through shared memory; a negative start ends the
// CTA's work):
//  a.ctl == nullptr (deterministic): CTA k owns rows [k*R/P, (k+1)*R/P), a function of
//    (R, P) only, so its partial -- and the fixed-order finish -- are bit-reproducible.
//  a.ctl != nullptr (non-deterministic): CTA k owns a fixed prefix of Ns stages, rows
//    [k*Ns*G, (k+1)*Ns*G), and the last ~2 stages' worth of rows a CTA would own, rows
//    [P*Ns*G, R), form a pool handed out G rows at a time by the counter a.ctl[1]: a CTA
//    that is done with its prefix early takes more of the tail, so none idles while
//    another still holds a queue.  CTA 0 opens the pool (sets the counter, then publishes
//    the call's tag in a.ctl[0]) before its own rows; a CTA that reaches the pool before
//    it is open takes nothing from it, and CTA 0 itself always drains it, so no CTA ever
//    waits on another.  Below 8*S stages a CTA (S the ring depth) the partition is the
//    deterministic one and the pool stays shut: when the pool runs dry every CTA still
//    holds S staged chunks, taken a ring's depth before it reaches them, and over so few
//    stages that spreads the CTAs' ends more than the pool evens them out (measured at
//    H=1536, 26 stages a CTA, S=4: 1.7 us behind the deterministic chunks).
// Either way CTA k writes its dw partial to a.part[k], and dx does not depend on the
// partition.
template <int VPT, int kCls, bool kFp32W, bool kDh, bool kRc>
__global__ void __launch_bounds__(bwd_max_threads(kCls, VPT), bwd_design_blocks_per_sm(kCls))
    rmsn_bwd_rows_kernel(const BwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NT = kDh ? 3 : 2;  // staged tensors: x, dy [, dh]
  const int H = a.map.H;
  const int NV = H >> 3;
  const int G = a.groups, NTg = a.ntg, S = a.stages;
  const int NW = NTg >> 5;
  const size_t stage_elems = static_cast<size_t>(NT) * G * H;
  const bool red_smem = NTg >= 32;  // else sub-warp groups: shuffles only
  constexpr bool kWSmem = bwd_w_in_smem(kCls, VPT);
  // kTm: each consumer thread's dw sums and compensation terms live in tensor memory (16
  // columns of its lane a vector) and come to registers one vector at a time
  constexpr bool kTm = kCls == kBwdTm;
  const SmemLayout L =
      smem_layout(S, NT, G, H, red_smem ? G : 0, G, kWSmem ? H : 0, 2 * S);

  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  uint64_t* redb = reinterpret_cast<uint64_t*>(smem + L.redb);  // [kRedBufs][G]
  float* slots = reinterpret_cast<float*>(smem + L.slots);       // [kRedBufs][G][32]
  float* rs_ring = reinterpret_cast<float*>(smem + L.rs);        // [S][RSP] staged rstd
  const int RSP = rs_stride(G);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  // [S][2]: each staged chunk's rows [start, end)
  volatile int32_t* srow = reinterpret_cast<volatile int32_t*>(smem + L.srow);

  const int tid = threadIdx.x;
  const int ncons = G * NTg;
  const int32_t k = blockIdx.x;
  uint32_t* tm_slot = reinterpret_cast<uint32_t*>(smem + L.abort_flag) + 2;
  const uint32_t tm_ncols = kTm ? tmem_alloc_cols(bwd_tm_cols(ncons / 32, VPT)) : 0u;

  if (tid >= ncons) {  // the producer warp (consumer warp 0 takes the tensor memory)
    init_row_barriers_warp(full, empty, S, static_cast<uint32_t>(G * NTg / 32), redb,
                           red_smem ? kRedBufs * G : 0, static_cast<uint32_t>(NW), tid - ncons);
    if (tid == ncons) *abort_flag = 0;
  }
  if constexpr (kTm) {
    // consumer warp 0 takes the columns (one CTA an SM: nothing else holds them); the
    // address reaches the other warps through shared memory
    if (tid < 32) {
      __syncwarp();  // the .sync.aligned tcgen05 forms want the whole warp converged
      tmem_alloc_warp(tm_slot, tm_ncols);
      tmem_fence_before_sync();
    }
  }
  __syncthreads();
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  if (tid >= ncons) {  // ---- producer warp ----
    if (tid == ncons) {
      const uint64_t pol = l2_evict_first_policy();
      const bool rs_bulk = !kRc && (reinterpret_cast<uintptr_t>(a.rstd) & 15u) == 0;
      const RowMap m{a.map.nh, H, a.map.s_tok, a.map.s_head};
      // rows [ra, rb) into slot s: x (strided), dy [, dh], and their rstd
      auto issue = [&](int s, int32_t ra, int32_t rb) {
        // The stage's rstd values travel with it, so no consumer waits on a global load:
        // the whole 16-byte blocks of rstd covering rows [ra, rb) by one bulk copy (slot
        // index r - a4), and rows past the last whole block of the array -- or every row,
        // when rstd is not 16-byte aligned -- by 4-byte async copies that the same
        // barrier tracks (one extra pending arrival, taken before the arrival below).
        // (kRc: no rstd to stage.)
        const int32_t a4 = ra & ~3;
        const int32_t b4 = kRc ? a4 : (rs_bulk ? min((rb + 3) & ~3, a.R & ~3) : a4);
        float* rsd = rs_ring + s * RSP;
        if (!kRc && rb > b4) {
          for (int32_t r = max(ra, b4); r < rb; ++r) cp_async_4(rsd + (r - a4), a.rstd + r);
          cp_async_mbar_arrive(&full[s]);
        }
        const uint32_t rs_bytes = static_cast<uint32_t>(b4 - a4) * 4u;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rb - ra) * H * 2u * NT + rs_bytes);
        if (rs_bytes) bulk_g2s(rsd, a.rstd + a4, rs_bytes, &full[s], pol);
        __nv_bfloat16* dst = ring + s * stage_elems;
        if (a.contig)
          copy_rows_contig(dst, a.x, H, ra, rb, &full[s], pol);
        else
          copy_rows(dst, a.x, m, ra, rb, &full[s], pol);
        copy_rows_contig(dst + G * H, a.dy, H, ra, rb, &full[s], pol);
        if constexpr (kDh) copy_rows_contig(dst + 2 * G * H, a.dh, H, ra, rb, &full[s], pol);
      };
      int32_t j = 0;  // stages whose full barrier has been armed
      const uint32_t R = static_cast<uint32_t>(a.R);
      const uint32_t per = static_cast<uint32_t>(a.P) * static_cast<uint32_t>(G);
      const uint32_t nfull = R / per;          // whole stages every CTA could own
      uint32_t pa, pb, pool;                   // this CTA's own rows [pa, pb), pool start
      if (nfull >= 8u * static_cast<uint32_t>(S) && a.ctl != nullptr) {  // prefix and pool
        const uint32_t Ns = nfull - 2;
        pa = static_cast<uint32_t>(k) * Ns * G;
        pb = pa + Ns * G;
        pool = per * Ns;
      } else {
        pa = static_cast<uint32_t>(r0_det(k, a.R, a.P));
        pb = static_cast<uint32_t>(r0_det(k + 1, a.R, a.P));
        pool = R;
      }
      if (k == 0 && pool < R) {  // open the pool: the counter first, then the tag
        a.ctl[1] = pool;
        __threadfence();
        st_release_u32(a.ctl, a.tag);
      }
      bool tail = false;
      uint32_t next = pa;
      uint32_t first_tail = R;  // the first pool chunk, taken while the prefix's last
                                // stage is issued (so its round trip is hidden too)
      for (;; ++j) {
        const int s = j % S;
        if (j >= S &&
            !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((j / S) - 1) & 1u, abort_flag,
                               a.err, kErrProducerWait))
          break;
        if (!tail && next >= pb) {  // prefix done: on to the pool
          tail = true;
          next = first_tail;
        }
        const uint32_t ra = next;
        if (ra >= R) {  // no rows left: an empty stage tells the consumers to stop
          srow[2 * s] = -1;
          mbar_arrive(&full[s]);
          ++j;
          break;
        }
        // the next tail chunk is taken now, so the atomic's round trip overlaps the wait
        // for the next free slot
        const uint32_t rb = tail ? min(ra + G, R) : min(ra + G, pb);
        if (!tail && rb >= pb && pool < R && ld_acquire_u32(a.ctl) == a.tag)
          first_tail = atomicAdd(a.ctl + 1, G);  // the pool is open: reserve a chunk
        next = tail ? atomicAdd(a.ctl + 1, G) : rb;
        srow[2 * s] = static_cast<int32_t>(ra);  // published by the arrival in issue()
        srow[2 * s + 1] = static_cast<int32_t>(rb);
        issue(s, static_cast<int32_t>(ra), static_cast<int32_t>(rb));
      }
      mbar_drain(full, S, j);
    }
    return;
  }

  // ---- consumers: group g, thread lt owns column vectors c = lt + v*NTg ----
  //
  // Split-phase rows: phase A of row j forms each warp's partial of sum_j (dy*w)*x and
  // arrives on the row's reduction mbarrier; phase B of row j-1 waits on that barrier
  // (normally long complete), re-reads row j-1 from shared memory, and produces dx and
  // the dw contributions.  Across rows a thread keeps only its columns' dw state and
  // weight in registers (the 4-vector multi-group build reads the weight from shared
  // memory instead).
  const int g = tid / NTg;
  const int lt = tid - g * NTg;
  const int wg = lt >> 5, lane = tid & 31;
  f2 wv[kWSmem ? 1 : VPT][4];  // the weight of this thread's columns (registers)
  f2 acc[VPT][4], cmp[VPT][4];  // (kTm: filled from tensor memory after the loop)
  float* wsm = reinterpret_cast<float*>(smem + L.w);  // or FP32 in shared memory
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = lt + v * NTg;
    if constexpr (!kWSmem) {
      if (c < NV) load_w8_pairs<kFp32W>(a.w, c, wv[v]);
    }
    if constexpr (!kTm) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[v][q] = f2_splat(0.f);
        cmp[v][q] = f2_splat(0.f);
      }
    }
  }
  // this thread's cells: vector v's 8 sums at columns tm + 16v .. +7, its 8 compensation
  // terms at +8 .. +15 (warps sharing a lane quadrant side by side)
  uint32_t tm = 0;
  if constexpr (kTm) {
    __syncwarp();
    tmem_fence_after_sync();
    const uint32_t w = static_cast<uint32_t>(tid >> 5);
    tm = tmem_warp_addr(*tm_slot, w, (w >> 2) * 16u * VPT);
    float z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) tmem_st16(tm + 16u * v, z);
  }
  if constexpr (kWSmem) {
    for (int c = tid; c < NV; c += ncons) {
      f2 p[4];
      load_w8_pairs<kFp32W>(a.w, c, p);
      // two planes of float4 (columns 0-3 and 4-7 of each vector), so that a warp's
      // reads of one plane are contiguous and free of bank conflicts
      float4* d = reinterpret_cast<float4*>(wsm);
      d[c] = make_float4(f2_lo(p[0]), f2_hi(p[0]), f2_lo(p[1]), f2_hi(p[1]));
      d[NV + c] = make_float4(f2_lo(p[2]), f2_hi(p[2]), f2_lo(p[3]), f2_hi(p[3]));
    }
    named_bar_sync(14, ncons);
  }
  // this thread's weight pairs for column vector c (its v-th)
  // shared-window addresses: the ring, and the weight planes
  const uint32_t ring32 = smem_u32(smem);
  const uint32_t w32 = ring32 + static_cast<uint32_t>(L.w);
  const uint32_t dy_off = static_cast<uint32_t>(G) * H * 2u;  // dy rows after x's in a stage
  auto wvec = [&](int v, int c, f2 (&p)[4]) {
    if constexpr (kWSmem) {
      const float4 a4 = lds128f_at(w32 + 16u * c);
      const float4 b4 = lds128f_at(w32 + 16u * (NV + c));
      p[0] = f2_make(a4.x, a4.y);
      p[1] = f2_make(a4.z, a4.w);
      p[2] = f2_make(b4.x, b4.y);
      p[3] = f2_make(b4.z, b4.w);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) p[q] = wv[v][q];
    }
  };
  const float inv_h = 1.0f / static_cast<float>(H);
  const float hf = static_cast<float>(H);
  // Phase A of group g's row in slot s (valid: the row exists): its share of
  // sum (dy*w)*x (and, kRc, of sum x^2), reduced over the group (sub-warp groups: returned;
  // whole-warp groups: published to the row's reduction slots).
  auto phase_a = [&](int32_t j, int s, bool valid) -> RowSums {
    const uint32_t st = ring32 + 2u * static_cast<uint32_t>(s * stage_elems + g * H);
    f2 dot0 = f2_splat(0.f), dot1 = f2_splat(0.f);
    f2 ss0 = f2_splat(0.f), ss1 = f2_splat(0.f);
    if (valid) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = lt + v * NTg;
        if (c < NV) {
          const uint4 xv = lds128_at(st + 16u * c);
          const uint4 dv = lds128_at(st + dy_off + 16u * c);
          f2 wl[4];
          wvec(v, c, wl);
          // (dy*x)*w: dy*x exact from the BF16 words, one rounding in the fma with w
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const f2 dyx = bf2_mul_exact(u4_get(dv, q), u4_get(xv, q));
            if (q & 1) {
              dot1 = f2_fma(dyx, wl[q], dot1);
              if constexpr (kRc) ss1 = bf2_sq_acc(u4_get(xv, q), ss1);
            } else {
              dot0 = f2_fma(dyx, wl[q], dot0);
              if constexpr (kRc) ss0 = bf2_sq_acc(u4_get(xv, q), ss0);
            }
          }
        }
      }
    }
    const f2 dsum = f2_add(dot0, dot1);
    const float part = f2_lo(dsum) + f2_hi(dsum);
    float spart = 0.f;
    if constexpr (kRc) {
      const f2 qsum = f2_add(ss0, ss1);
      spart = f2_lo(qsum) + f2_hi(qsum);
    }
    if (red_smem) {
      // slot row of 32 floats: the warps' sums of (dy*w)*x in [0, NW), of x^2 in
      // [16, 16 + NW) (at most 12 warps a group)
      const float dot = warp_allsum(part);
      float ssw = 0.f;
      if constexpr (kRc) ssw = warp_allsum(spart);
      if (lane == 0) {
        float* sl = slots + ((j % kRedBufs) * G + g) * 32;
        sl[wg] = dot;
        if constexpr (kRc) sl[16 + wg] = ssw;
        mbar_arrive(&redb[(j % kRedBufs) * G + g]);
      }
      return RowSums{0.f, 0.f};
    }
    RowSums r{subwarp_allsum(part, NTg), 0.f};
    if constexpr (kRc) r.ss = subwarp_allsum(spart, NTg);
    return r;
  };
  // Phase B of stage jj (slot s, first row stage_ra): dx and the dw contributions.
  auto phase_b = [&](int32_t jj, int s, int32_t stage_ra, int32_t row_end, RowSums sums) {
    const int32_t row = stage_ra + g;
    float dot = sums.dot, ss = sums.ss;
    if (red_smem) {
      const int rb = (jj % kRedBufs) * G + g;
      mbar_wait_bounded(&redb[rb], static_cast<uint32_t>(jj / kRedBufs) & 1u, abort_flag, a.err,
                        kErrConsumerWait);
      dot = slot_sum(slots + rb * 32, NW);
      if constexpr (kRc) ss = slot_sum(slots + rb * 32 + 16, NW);
    }
    const bool rv = row < row_end;
    // (kTm: every thread of the warp takes part in the tensor-memory traffic, with or
    // without a row)
    if (kTm || rv) {
      // this row's rstd: staged with the row (the stage is held until phase B ends), or
      // (kRc) recomputed from the row's sum of squares the way the forward forms it
      float rs = 0.f;
      if (rv) {
        if constexpr (kRc) {
          rs = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, hf), a.eps));
          if (a.rstd_out != nullptr && lt == 0) a.rstd_out[row] = rs;
        } else {
          rs = rs_ring[s * RSP + (row - (stage_ra & ~3))];
        }
      }
      // rstd = rs_hi + rs_lo with rs_hi holding rstd's top 8 significant bits: dy*x has
      // at most 16 significant bits (two BF16 significands), so dy*x*rs_hi is exact in
      // FP32, and dy*x*rs_lo, 2^-8 smaller, only feeds the compensation term.
      const float rs_hi = __uint_as_float(__float_as_uint(rs) & 0xffff0000u);
      const f2 rs2 = f2_splat(rs), rh2 = f2_splat(rs_hi);
      // c = (1/H) sum g*xhat = (rstd/H) sum (dy*w)*x
      // dx = rstd*(g - x*(c*rstd)): xhat*c as one product of x, so the cancelling pair
      // is a single fma; c*rstd is on the scale of dx, so no new overflow or underflow
      const f2 ncr2 = f2_splat(-(dot * (rs * inv_h)) * rs);
      const uint32_t st = ring32 + 2u * static_cast<uint32_t>(s * stage_elems + g * H);
      const size_t out_row = static_cast<size_t>(row) * H;
      if constexpr (kTm) {
        __syncwarp();
        tmem_wait_st();  // the previous row's sums are stored before they are loaded
      }
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = lt + v * NTg;
        const bool live = rv && c < NV;
        float tv[16];  // kTm: this vector's sums [0, 8) and compensation terms [8, 16)
        if constexpr (kTm) tmem_ld16(tm + 16u * v, tv);
        f2 dyx[4];
        if (live) {
          const uint4 xv = lds128_at(st + 16u * c);
          const uint4 dv = lds128_at(st + dy_off + 16u * c);
          uint4 hv = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (kDh) hv = lds128_at(st + 2u * dy_off + 16u * c);
          f2 wl[4];
          wvec(v, c, wl);
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const f2 x2 = bf2_to_f2(u4_get(xv, q));
            const f2 d2 = bf2_to_f2(u4_get(dv, q));
            const f2 gw = f2_mul(d2, wl[q]);
            f2 d = f2_mul(f2_fma(x2, ncr2, gw), rs2);  // (g - xhat*c) * rstd
            if constexpr (kDh) d = f2_add(d, bf2_to_f2(u4_get(hv, q)));
            o[q] = f2_to_bf2(d);
            dyx[q] = f2_mul(d2, x2);
            if constexpr (!kTm) {
              // dw: running sum of the exact products dy*x*rs_hi with a Fast2Sum
              // compensation term, which also collects dy*x*rs_lo.  t = acc + p in one
              // fma (p is exact); acc - t is exact (Fast2Sum), so dy*x*rs + (acc - t) is
              // the addition's error plus dy*x*rs_lo, rounded once
              const f2 t = f2_fma(dyx[q], rh2, acc[v][q]);
              cmp[v][q] = f2_add(cmp[v][q], f2_fma(dyx[q], rs2, f2_sub(acc[v][q], t)));
              acc[v][q] = t;
            }
          }
          stg128(a.dx + out_row + c * 8, make_uint4(o[0], o[1], o[2], o[3]));
        }
        if constexpr (kTm) {
          __syncwarp();
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // the same update, on the loaded cells
              const f2 av = f2_make(tv[2 * q], tv[2 * q + 1]);
              const f2 t = f2_fma(dyx[q], rh2, av);
              const f2 cv = f2_add(f2_make(tv[8 + 2 * q], tv[9 + 2 * q]),
                                   f2_fma(dyx[q], rs2, f2_sub(av, t)));
              tv[2 * q] = f2_lo(t);
              tv[2 * q + 1] = f2_hi(t);
              tv[8 + 2 * q] = f2_lo(cv);
              tv[9 + 2 * q] = f2_hi(cv);
            }
          }
          __syncwarp();
          tmem_st16(tm + 16u * v, tv);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
  };

  // Stages in the order the producer filled them; a negative chunk start (or an
  // abort) ends the loop, warp-uniformly (every lane reads the same start).
  RowSums carry{0.f, 0.f};
  int32_t ra_prev = 0, rb_prev = 0;
  // slot and parity of stage j, and the slot of stage j-1, kept by increments (no
  // division by the runtime ring depth on the per-row path)
  int s = 0, s_prev = 0;
  uint32_t ph = 0;
  for (int32_t j = 0;; ++j) {
    const bool ok = mbar_wait_bounded(&full[s], ph, abort_flag, a.err, kErrConsumerWait);
    const int32_t ra = ok ? srow[2 * s] : -1;
    const int32_t rb = ok ? srow[2 * s + 1] : -1;
    const bool stop = __any_sync(0xffffffffu, ra < 0);
    RowSums cur{0.f, 0.f};
    if (!stop) cur = phase_a(j, s, ra + g < rb);
    if (j >= 1) phase_b(j - 1, s_prev, ra_prev, rb_prev, carry);
    if (stop) break;
    ra_prev = ra;
    rb_prev = rb;
    carry = cur;
    s_prev = s;
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }

  if constexpr (kTm) {
    // the sums come back to registers, and warp 0 frees the columns once every consumer
    // has loaded its own
    __syncwarp();
    tmem_wait_st();
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      float tv[16];
      tmem_ld16(tm + 16u * v, tv);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[v][q] = f2_make(tv[2 * q], tv[2 * q + 1]);
        cmp[v][q] = f2_make(tv[8 + 2 * q], tv[9 + 2 * q]);
      }
    }
    tmem_fence_before_sync();
    named_bar_sync(13, ncons);
    if (tid < 32) {
      __syncwarp();
      tmem_fence_after_sync();
      tmem_dealloc_warp(*tm_slot, tm_ncols);
    }
  }

  // ---- this CTA's dw partial: (hi, lo) with hi + lo == acc + cmp exactly ----
  float* part = a.part + static_cast<size_t>(k) * 2 * H;
  if (G == 1) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = lt + v * NTg;
      if (c < NV) {
        f2 hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hi[q] = f2_add(acc[v][q], cmp[v][q]);
          lo[q] = f2_sub(cmp[v][q], f2_sub(hi[q], acc[v][q]));
        }
        ulonglong2* ph = reinterpret_cast<ulonglong2*>(part + c * 8);
        ulonglong2* pl = reinterpret_cast<ulonglong2*>(part + H + c * 8);
        ph[0] = make_ulonglong2(hi[0].v, hi[1].v);
        ph[1] = make_ulonglong2(hi[2].v, hi[3].v);
        pl[0] = make_ulonglong2(lo[0].v, lo[1].v);
        pl[1] = make_ulonglong2(lo[2].v, lo[3].v);
      }
    }
  } else {
    // several row groups: combine them through shared memory in group order.  The ring
    // is free once every consumer is past its loop: each stage was waited on (full) by
    // every group that had a row in it before that group finished.
    named_bar_sync(15, ncons);
    // cb: [G][2][H] (hi, lo), each H-slab stored as two planes of float4 (columns 0-3 and
    // 4-7 of every vector) so that a warp's stores of one plane are contiguous
    float* cb = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = lt + v * NTg;
      if (c < NV) {
        f2 hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hi[q] = f2_add(acc[v][q], cmp[v][q]);
          lo[q] = f2_sub(cmp[v][q], f2_sub(hi[q], acc[v][q]));
        }
        ulonglong2* ph = reinterpret_cast<ulonglong2*>(cb + (2 * g) * H);
        ulonglong2* pl = reinterpret_cast<ulonglong2*>(cb + (2 * g + 1) * H);
        ph[c] = make_ulonglong2(hi[0].v, hi[1].v);
        ph[NV + c] = make_ulonglong2(hi[2].v, hi[3].v);
        pl[c] = make_ulonglong2(lo[0].v, lo[1].v);
        pl[NV + c] = make_ulonglong2(lo[2].v, lo[3].v);
      }
    }
    named_bar_sync(15, ncons);
    // Per column: TwoSum of the groups' hi in group order, their lo and the errors summed
    // beside.  Where that keeps at least half the consumers busy, a thread takes one
    // float4 of a plane (u < NV: columns 8u..8u+3; else columns 8(u-NV)+4..+7), four
    // independent columns; otherwise (narrow rows, many groups) a column a thread.
    // Either way the slabs' loads are issued ahead of the additions.
    if (H < 2 * ncons) {
      for (int col = tid; col < H; col += ncons) {
        const int at = ((col & 7) >> 2) * (4 * NV) + (col >> 3) * 4 + (col & 3);
        float sacc = 0.f, e = 0.f;
#pragma unroll 4
        for (int gi = 0; gi < G; ++gi) {
          float err;
          sacc = two_sum(sacc, cb[(2 * gi) * H + at], err);
          e = __fadd_rn(e, __fadd_rn(err, cb[(2 * gi + 1) * H + at]));
        }
        const float hi = __fadd_rn(sacc, e);
        part[col] = hi;
        part[H + col] = __fsub_rn(e, __fsub_rn(hi, sacc));
      }
    } else {
      const float4* cb4 = reinterpret_cast<const float4*>(smem);
      const int slab4 = H / 4;  // float4s a slab
      for (int u = tid; u < 2 * NV; u += ncons) {
        const int col0 = u < NV ? 8 * u : 8 * (u - NV) + 4;
        float sacc[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int gi = 0; gi < G; ++gi) {
          const float4 h4 = cb4[(2 * gi) * slab4 + u];
          const float4 l4 = cb4[(2 * gi + 1) * slab4 + u];
          const float hv[4] = {h4.x, h4.y, h4.z, h4.w};
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float err;
            sacc[i] = two_sum(sacc[i], hv[i], err);
            e[i] = __fadd_rn(e[i], __fadd_rn(err, lv[i]));
          }
        }
        float hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          hi[i] = __fadd_rn(sacc[i], e[i]);
          lo[i] = __fsub_rn(e[i], __fsub_rn(hi[i], sacc[i]));
        }
        *reinterpret_cast<float4*>(part + col0) = make_float4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<float4*>(part + H + col0) = make_float4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  }
}

// The kernel build for a launch shape (both modes), per kRc; each value's translation unit
// instantiates only its own builds.  (bwd_shape gives 1-vector lanes the narrow class, 2-
// and 4-vector threads the multi, tensor-memory or wide class, 3-vector threads the multi
// or tensor-memory class.)
template <bool kRc>
const void* pick_rows_kernel(const Shape& s, bool fp32w, bool dh) {
  auto fn = [](auto k) { return reinterpret_cast<const void*>(k); };
#define RMSN_PICK(V, C)                                                               \
  (fp32w ? (dh ? fn(&rmsn_bwd_rows_kernel<V, C, true, true, kRc>)                     \
               : fn(&rmsn_bwd_rows_kernel<V, C, true, false, kRc>))                   \
         : (dh ? fn(&rmsn_bwd_rows_kernel<V, C, false, true, kRc>)                    \
               : fn(&rmsn_bwd_rows_kernel<V, C, false, false, kRc>)))
  if (s.cls == kBwdTm)
    return s.vpt == 2 ? RMSN_PICK(2, kBwdTm)
                      : (s.vpt == 3 ? RMSN_PICK(3, kBwdTm) : RMSN_PICK(4, kBwdTm));
  if (s.vpt == 1) return RMSN_PICK(1, kBwdNarrow);
  if (s.vpt == 2) return s.cls == kBwdMulti ? RMSN_PICK(2, kBwdMulti) : RMSN_PICK(2, kBwdWide);
  if (s.vpt == 3) return RMSN_PICK(3, kBwdMulti);
  return s.cls == kBwdMulti ? RMSN_PICK(4, kBwdMulti) : RMSN_PICK(4, kBwdWide);
#undef RMSN_PICK
}

}  // namespace rmsn
