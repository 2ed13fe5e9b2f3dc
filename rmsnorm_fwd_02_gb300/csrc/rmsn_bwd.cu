// rmsn_bwd.cu -- RMSNorm training backward for sm_103a: dx row pass fused with the dw
// partial sums, and the fixed-order dw finish.
//
// Per normalized row, with r the forward's rstd (flashinfer PR #8827, description: the
// backward's BF16 dx and FP32 dw; the residual form's combined gradient):
//   xhat_j = x_j * r,  g_j = dy_j * w_j,  c = (1/H) sum_j g_j * xhat_j
//        = (r/H) * sum_j (dy_j * w_j) * x_j
//   dx_j   = BF16((g_j - xhat_j * c) * r  [+ dh_j])
//   dw_j  += dy_j * xhat_j          over every row of every CTA's chunk
//
// dw accuracy (PR #8849 and PR #8827's route notes: every dw element within
// atol 1e-4 + rtol 1e-4 of an FP64 sum, a budget plain FP32 running sums break at large
// T).  Two error sources are removed: the rounding of each product and the rounding of
// each addition.  With rstd split as rs_hi (its top 8 significant bits) + rs_lo, the
// product dy*x*rs_hi is exact in FP32 (dy*x carries at most 16 significant bits), and
// dy*x*rs_lo is 2^-8 smaller.  Each consumer thread keeps per column a running FP32 sum
// of the exact products and a compensation term that collects each addition's Fast2Sum
// error plus the small dy*x*rs_lo terms.  A CTA writes its chunk's partial as an
// unevaluated (hi, lo) FP32 pair per column; the finish kernel adds the P pairs in a
// fixed order with Knuth's TwoSum.  What remains is about the final rounding of dw to
// FP32.  The row -> CTA chunk mapping is fixed by (R, P) and the finish order by P, so dw
// is bit-reproducible whenever P is; dx does not depend on P at all.
//
// Split-phase rows (see the consumer loop) keep the row reduction off the critical path.
// Arithmetic runs on packed FP32 pairs (f32x2): two columns per instruction.
#include "rmsn_common.cuh"
#include "rmsn_launch.h"

namespace rmsn {

// Knuth's TwoSum: s + err == a + b exactly, no ordering assumption.
__device__ __forceinline__ float two_sum(float a, float b, float& err) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bp);
  err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
  return s;
}

// Launch bounds per shape class (rmsn_launch.h): narrow CTAs of up to 256 consumers, two
// an SM; multi-group CTAs of up to 480 consumers and wide CTAs (384 consumers with
// 2-vector threads, 256 with 4-vector threads), one an SM; each + the producer warp.
template <int VPT, int kCls, bool kFp32W, bool kDh>
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
  const SmemLayout L = smem_layout(S, NT, G, H, red_smem ? G : 0, G, kWSmem ? H : 0);

  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  uint64_t* redb = reinterpret_cast<uint64_t*>(smem + L.redb);  // [kRedBufs][G]
  float* slots = reinterpret_cast<float*>(smem + L.slots);       // [kRedBufs][G][32]
  float* rs_ring = reinterpret_cast<float*>(smem + L.rs);        // [S][RSP] staged rstd
  const int RSP = rs_stride(G);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

  const int tid = threadIdx.x;
  const int ncons = G * NTg;
  const int32_t k = blockIdx.x;
  const int32_t r0 = static_cast<int32_t>((static_cast<int64_t>(k) * a.R) / a.P);
  const int32_t r1 = static_cast<int32_t>((static_cast<int64_t>(k + 1) * a.R) / a.P);
  const int32_t nstage = (r1 - r0 + G - 1) / G;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], static_cast<uint32_t>(G * NTg / 32));  // one arrival per warp
    }
    if (red_smem)
      for (int i = 0; i < kRedBufs * G; ++i) mbar_init(&redb[i], static_cast<uint32_t>(NW));
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  if (tid >= ncons) {  // ---- producer warp ----
    if (tid == ncons) {
      const uint64_t pol = l2_evict_first_policy();
      const bool rs_bulk = (reinterpret_cast<uintptr_t>(a.rstd) & 15u) == 0;
      const RowMap m{a.map.nh, H, a.map.s_tok, a.map.s_head};
      int32_t j = 0;
      for (; j < nstage; ++j) {
        const int s = j % S;
        if (j >= S &&
            !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((j / S) - 1) & 1u, abort_flag,
                               a.err, kErrProducerWait))
          break;
        const int32_t ra = r0 + j * G;
        const int32_t rb = min(ra + G, r1);
        // The stage's rstd values travel with it, so no consumer waits on a global load:
        // the whole 16-byte blocks of rstd covering rows [ra, rb) by one bulk copy (slot
        // index r - a4), and rows past the last whole block of the array -- or every row,
        // when rstd is not 16-byte aligned -- by 4-byte async copies that the same
        // barrier tracks (one extra pending arrival, taken before the arrival below).
        const int32_t a4 = ra & ~3;
        const int32_t b4 = rs_bulk ? min((rb + 3) & ~3, a.R & ~3) : a4;
        float* rsd = rs_ring + s * RSP;
        if (rb > b4) {
          for (int32_t r = max(ra, b4); r < rb; ++r) cp_async_4(rsd + (r - a4), a.rstd + r);
          cp_async_mbar_arrive(&full[s]);
        }
        const uint32_t rs_bytes = static_cast<uint32_t>(b4 - a4) * 4u;
        mbar_arrive_expect_tx(&full[s],
                              static_cast<uint32_t>(rb - ra) * H * 2u * NT + rs_bytes);
        if (rs_bytes) bulk_g2s(rsd, a.rstd + a4, rs_bytes, &full[s], pol);
        __nv_bfloat16* dst = ring + s * stage_elems;
        if (a.contig)
          copy_rows_contig(dst, a.x, H, ra, rb, &full[s], pol);
        else
          copy_rows(dst, a.x, m, ra, rb, &full[s], pol);
        copy_rows_contig(dst + G * H, a.dy, H, ra, rb, &full[s], pol);
        if constexpr (kDh) copy_rows_contig(dst + 2 * G * H, a.dh, H, ra, rb, &full[s], pol);
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
  f2 acc[VPT][4], cmp[VPT][4];
  float* wsm = reinterpret_cast<float*>(smem + L.w);  // or FP32 in shared memory
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = lt + v * NTg;
    if constexpr (!kWSmem) {
      if (c < NV) load_w8_pairs<kFp32W>(a.w, c, wv[v]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[v][q] = f2_splat(0.f);
      cmp[v][q] = f2_splat(0.f);
    }
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
  auto wvec = [&](int v, int c, f2 (&p)[4]) {
    if constexpr (kWSmem) {
      const float4 a4 = reinterpret_cast<const float4*>(wsm)[c];
      const float4 b4 = reinterpret_cast<const float4*>(wsm)[NV + c];
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
  // Rows of this warp's first group: every lane of a warp runs the same iterations (the
  // shuffles need them all); groups past the chunk's end skip the row work.
  const int g0 = red_smem ? g : (tid & ~31) / NTg;
  const int32_t ng = (r1 - r0 > g0) ? (r1 - r0 - g0 + G - 1) / G : 0;

  float dot_carry = 0.f; // sub-warp groups: row j-1's sum of (dy*w)*x
  for (int32_t j = 0; j <= ng; ++j) {
    float dot_new = 0.f;
    // ---- phase A, row j: partial of sum (dy*w)*x ----
    if (j < ng) {
      const int32_t row = r0 + j * G + g;
      const bool valid = row < r1;
      const int s = j % S;
      mbar_wait_bounded(&full[s], static_cast<uint32_t>(j / S) & 1u, abort_flag, a.err,
                        kErrConsumerWait);
      const __nv_bfloat16* st = ring + s * stage_elems + static_cast<size_t>(g) * H;
      f2 dot0 = f2_splat(0.f), dot1 = f2_splat(0.f);
      if (valid) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
            const uint4 xv = lds128(st + c * 8);
            const uint4 dv = lds128(st + static_cast<size_t>(G) * H + c * 8);
            f2 wl[4];
            wvec(v, c, wl);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const f2 gw = f2_mul(bf2_to_f2(u4_get(dv, q)), wl[q]);
              if (q & 1)
                dot1 = f2_fma(gw, bf2_to_f2(u4_get(xv, q)), dot1);
              else
                dot0 = f2_fma(gw, bf2_to_f2(u4_get(xv, q)), dot0);
            }
          }
        }
      }
      const f2 dsum = f2_add(dot0, dot1);
      const float part = f2_lo(dsum) + f2_hi(dsum);
      if (red_smem) {
        const float dot = warp_allsum(part);
        if (lane == 0) {
          slots[((j % kRedBufs) * G + g) * 32 + wg] = dot;
          mbar_arrive(&redb[(j % kRedBufs) * G + g]);
        }
      } else {
        dot_new = subwarp_allsum(part, NTg);
      }
    }
    // ---- phase B, row j-1: dx and the dw contributions ----
    if (j >= 1) {
      const int32_t jj = j - 1;
      const int32_t row = r0 + jj * G + g;
      const int s = jj % S;
      float dot = dot_carry;
      if (red_smem) {
        const int rb = (jj % kRedBufs) * G + g;
        mbar_wait_bounded(&redb[rb], static_cast<uint32_t>(jj / kRedBufs) & 1u, abort_flag,
                          a.err, kErrConsumerWait);
        dot = slot_sum(slots + rb * 32, NW);
      }
      if (row < r1) {
        // this row's rstd, staged with the row (the stage is held until phase B ends)
        const float rs = rs_ring[s * RSP + (row - ((r0 + jj * G) & ~3))];
        // rstd = rs_hi + rs_lo with rs_hi holding rstd's top 8 significant bits: dy*x has
        // at most 16 significant bits (two BF16 significands), so dy*x*rs_hi is exact in
        // FP32, and dy*x*rs_lo, 2^-8 smaller, only feeds the compensation term.
        const float rs_hi = __uint_as_float(__float_as_uint(rs) & 0xffff0000u);
        const f2 rs2 = f2_splat(rs), rh2 = f2_splat(rs_hi);
        const f2 rl2 = f2_splat(__fsub_rn(rs, rs_hi));
        // c = (1/H) sum g*xhat = (rstd/H) sum (dy*w)*x
        // dx = rstd*(g - x*(c*rstd)): xhat*c as one product of x, so the cancelling pair
        // is a single fma; c*rstd is on the scale of dx, so no new overflow or underflow
        const f2 ncr2 = f2_splat(-(dot * (rs * inv_h)) * rs);
        const __nv_bfloat16* st = ring + s * stage_elems + static_cast<size_t>(g) * H;
        const size_t out_row = static_cast<size_t>(row) * H;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
            const uint4 xv = lds128(st + c * 8);
            const uint4 dv = lds128(st + static_cast<size_t>(G) * H + c * 8);
            uint4 hv = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (kDh) hv = lds128(st + static_cast<size_t>(2 * G) * H + c * 8);
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
              // dw: running sum of the exact products dy*x*rs_hi with a Fast2Sum
              // compensation term, which also collects dy*x*rs_lo
              const f2 dyx = f2_mul(d2, x2);
              const f2 p = f2_mul(dyx, rh2);
              const f2 t = f2_add(acc[v][q], p);
              const f2 e = f2_add(f2_sub(acc[v][q], t), p);
              cmp[v][q] = f2_fma(dyx, rl2, f2_add(cmp[v][q], e));
              acc[v][q] = t;
            }
            stg128(a.dx + out_row + c * 8, make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
    }
    dot_carry = dot_new;
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
    return;
  }
  // several row groups: combine them through shared memory in group order.  The ring is
  // free once every consumer is past its loop: each stage was waited on (full) by every
  // group that had a row in it before that group finished.
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
  for (int col = tid; col < H; col += ncons) {
    const int at = ((col & 7) >> 2) * (4 * NV) + (col >> 3) * 4 + (col & 3);
    float sacc = 0.f, e = 0.f;
    for (int gi = 0; gi < G; ++gi) {
      float err;
      sacc = two_sum(sacc, cb[(2 * gi) * H + at], err);
      e = __fadd_rn(e, __fadd_rn(err, cb[(2 * gi + 1) * H + at]));
    }
    const float hi = __fadd_rn(sacc, e);
    part[col] = hi;
    part[H + col] = __fsub_rn(e, __fsub_rn(hi, sacc));
  }
}

// dw[col] = sum over k = 0..P-1 of (hi_k + lo_k), in a fixed order: slice i of the
// kFinishSlices slices takes k in [i*P/slices, (i+1)*P/slices) in increasing k, then the
// slice sums are combined by a pairwise tree in slice order (i with i + stride, stride
// halving).  TwoSum carries the error terms throughout.  Each thread walks only ~P/32
// partials with four loads in flight, so the kernel is a short tail.
__global__ void __launch_bounds__(kFinishCols* kFinishSlices)
    rmsn_dw_finish_kernel(const float* __restrict__ part, float* __restrict__ dw, int P, int H) {
  __shared__ float sh[kFinishSlices][kFinishCols];
  __shared__ float se[kFinishSlices][kFinishCols];
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int cl = threadIdx.x % kFinishCols;
  const int sl = threadIdx.x / kFinishCols;
  const int col = blockIdx.x * kFinishCols + cl;
  float s = 0.f, e = 0.f;
  if (col < H) {
    const int ka = (sl * P) / kFinishSlices;
    const int kb = ((sl + 1) * P) / kFinishSlices;
    const float* p = part + static_cast<size_t>(ka) * 2 * H + col;
    int kk = ka;
    for (; kk + 4 <= kb; kk += 4, p += static_cast<size_t>(8) * H) {
      float hi[4], lo[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        hi[u] = p[static_cast<size_t>(2 * u) * H];
        lo[u] = p[static_cast<size_t>(2 * u + 1) * H];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float err;
        s = two_sum(s, hi[u], err);
        e = __fadd_rn(e, __fadd_rn(err, lo[u]));
      }
    }
    for (; kk < kb; ++kk, p += static_cast<size_t>(2) * H) {
      float err;
      s = two_sum(s, p[0], err);
      e = __fadd_rn(e, __fadd_rn(err, p[H]));
    }
  }
  sh[sl][cl] = s;
  se[sl][cl] = e;
  __syncthreads();
#pragma unroll
  for (int stride = kFinishSlices / 2; stride > 0; stride >>= 1) {
    if (sl < stride) {
      float err;
      const float S = two_sum(sh[sl][cl], sh[sl + stride][cl], err);
      se[sl][cl] = __fadd_rn(__fadd_rn(se[sl][cl], se[sl + stride][cl]), err);
      sh[sl][cl] = S;
    }
    __syncthreads();
  }
  if (sl == 0 && col < H) dw[col] = __fadd_rn(sh[0][cl], se[0][cl]);
}

template <int VPT, int kCls, bool kFp32W, bool kDh>
static const void* bwd_kernel_ptr() {
  return reinterpret_cast<const void*>(&rmsn_bwd_rows_kernel<VPT, kCls, kFp32W, kDh>);
}

template <int VPT, int kCls>
static const void* pick_bwd_v(bool fp32w, bool dh) {
  if (fp32w)
    return dh ? bwd_kernel_ptr<VPT, kCls, true, true>() : bwd_kernel_ptr<VPT, kCls, true, false>();
  return dh ? bwd_kernel_ptr<VPT, kCls, false, true>() : bwd_kernel_ptr<VPT, kCls, false, false>();
}

static const void* pick_bwd(const Shape& s, bool fp32w, bool dh) {
  if (s.vpt == 1) return pick_bwd_v<1, kBwdNarrow>(fp32w, dh);
  if (s.vpt == 2) {
    if (s.cls == kBwdMulti) return pick_bwd_v<2, kBwdMulti>(fp32w, dh);
    if (s.cls == kBwdWide) return pick_bwd_v<2, kBwdWide>(fp32w, dh);
    return pick_bwd_v<2, kBwdNarrow>(fp32w, dh);
  }
  if (s.vpt == 3) return pick_bwd_v<3, kBwdMulti>(fp32w, dh);
  if (s.cls == kBwdMulti) return pick_bwd_v<4, kBwdMulti>(fp32w, dh);
  return pick_bwd_v<4, kBwdWide>(fp32w, dh);
}

cudaError_t prepare_kernel(const void* fn, size_t smem);
int blocks_per_sm(const void* fn, int threads, size_t smem);
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       void** args);

int bwd_blocks_per_sm(const Shape& s, bool fp32w) {
  return blocks_per_sm(pick_bwd(s, fp32w, s.tensors == 3), s.threads, s.smem);
}

cudaError_t launch_bwd_rows(const BwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st) {
  const void* fn = pick_bwd(s, fp32w, a.dh != nullptr);
  cudaError_t e = prepare_kernel(fn, s.smem);
  if (e != cudaSuccess) return e;
  BwdArgs copy = a;
  void* args[] = {&copy};
  return launch_pdl(fn, dim3(static_cast<unsigned>(a.P)), dim3(static_cast<unsigned>(s.threads)),
                    s.smem, st, args);
}

cudaError_t launch_dw_finish(const float* part, float* dw, int P, int H, cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&rmsn_dw_finish_kernel);
  void* args[] = {&part, &dw, &P, &H};
  const unsigned grid = static_cast<unsigned>((H + kFinishCols - 1) / kFinishCols);
  return launch_pdl(fn, dim3(grid), dim3(kFinishCols * kFinishSlices), 0, st, args);
}

}  // namespace rmsn
