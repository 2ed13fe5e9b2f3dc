// rmsn_small.cu -- the RMSNorm training backward for small inputs, in one launch.
//
// For at most kSmallMaxRows normalized rows the staged row pass and its separate dw
// finish are mostly fixed cost (two launches, the ring's first load, the partial write).
// This kernel does the whole backward in one launch and without a workspace, with two
// kinds of CTA:
//
//  - row tasks (blocks [0, Pr)): one row per group of gt threads, VPT 16-byte column
//    vectors a thread, every load of the row in flight at once; the group's sum of
//    (dy*w)*x is a warp butterfly and a fixed-order sum of the warp partials through
//    shared memory; dx uses the row pass's arithmetic (rmsn_bwd.cu), so the two paths
//    agree to the bit wherever their sums of (dy*w)*x do.
//  - column tasks (blocks [Pr, Pr + Pc)): block k owns the column vectors
//    [kSmallColVecs*k, kSmallColVecs*(k+1)); thread (v, sl) sums dy*x*rstd for its vector
//    over the rows sl, sl + kSmallSlices, ... in increasing order, with the row pass's
//    exact products and Fast2Sum compensation, and the kSmallSlices slices then combine
//    as (hi, lo) pairs by a pairwise TwoSum tree in slice order.
//
// Every order is fixed by (R, H), so dw is bit-reproducible in both modes.  (The pages'
// column-task kernel for small T has the same split of dw over columns; this one also
// carries the row tasks, so that one launch returns dx and dw.)
#include "rmsn_common.cuh"
#include "rmsn_launch.h"

namespace rmsn {

namespace {

// Knuth's TwoSum: s + err == a + b exactly.
__device__ __forceinline__ float two_sum_exact(float a, float b, float& err) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bp);
  err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
  return s;
}

constexpr int kSmallCols = kSmallColVecs * 8;

}  // namespace

template <int VPT, bool kFp32W, bool kDh>
__global__ void __launch_bounds__(kSmallThreads)
    rmsn_bwd_small_kernel(const BwdArgs a, float* __restrict__ dw, int Pr) {
  __shared__ __align__(16) float sm[2 * kSmallSlices * kSmallCols];
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int H = a.map.H;
  const int NV = H >> 3;
  const int tid = threadIdx.x;
  const int lane = tid & 31;

  if (static_cast<int>(blockIdx.x) < Pr) {
    // ---- row task ----
    const int per = (NV + VPT - 1) / VPT;
    const int gt = per <= 32 ? 32 : (per + 31) / 32 * 32;  // threads a row
    const int groups = kSmallThreads / gt;                  // rows a CTA
    const int g = tid / gt;
    const int lt = tid - g * gt;
    const int nw = gt >> 5;
    const int32_t row = static_cast<int32_t>(blockIdx.x) * groups + g;
    const bool live = g < groups && row < a.R;  // threads past groups*gt stay idle
    uint4 xv[VPT], dv[VPT];
    f2 wv[VPT][4];
    float part = 0.f;
    size_t xoff = 0;
    if (live) {
      const int32_t t = row / a.map.nh;
      const int32_t hd = row - t * a.map.nh;
      xoff = static_cast<size_t>(static_cast<int64_t>(t) * a.map.s_tok +
                                 static_cast<int64_t>(hd) * a.map.s_head);
      f2 dot0 = f2_splat(0.f), dot1 = f2_splat(0.f);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = lt + v * gt;
        xv[v] = dv[v] = make_uint4(0u, 0u, 0u, 0u);
        if (c < NV) {
          xv[v] = *reinterpret_cast<const uint4*>(a.x + xoff + c * 8);
          dv[v] = *reinterpret_cast<const uint4*>(a.dy + static_cast<size_t>(row) * H + c * 8);
          load_w8_pairs<kFp32W>(a.w, c, wv[v]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // (dy*x)*w, dy*x exact, as the row pass forms it
            const f2 dyx = bf2_mul_exact(u4_get(dv[v], q), u4_get(xv[v], q));
            if (q & 1)
              dot1 = f2_fma(dyx, wv[v][q], dot1);
            else
              dot0 = f2_fma(dyx, wv[v][q], dot0);
          }
        }
      }
      const f2 dsum = f2_add(dot0, dot1);
      part = f2_lo(dsum) + f2_hi(dsum);
    }
    const float wsum = warp_allsum(part);
    if (lane == 0) sm[tid >> 5] = wsum;  // one slot a warp; a group's warps are adjacent
    __syncthreads();
    if (!live) return;
    float dot = 0.f;
    for (int i = 0; i < nw; ++i) dot += sm[g * nw + i];
    const float rs = a.rstd[row];
    const float inv_h = 1.0f / static_cast<float>(H);
    const f2 rs2 = f2_splat(rs);
    const f2 ncr2 = f2_splat(-(dot * (rs * inv_h)) * rs);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = lt + v * gt;
      if (c < NV) {
        uint4 hv = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (kDh)
          hv = *reinterpret_cast<const uint4*>(a.dh + static_cast<size_t>(row) * H + c * 8);
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const f2 gw = f2_mul(bf2_to_f2(u4_get(dv[v], q)), wv[v][q]);
          f2 d = f2_mul(f2_fma(bf2_to_f2(u4_get(xv[v], q)), ncr2, gw), rs2);
          if constexpr (kDh) d = f2_add(d, bf2_to_f2(u4_get(hv, q)));
          o[q] = f2_to_bf2(d);
        }
        stg128(a.dx + static_cast<size_t>(row) * H + c * 8, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
    return;
  }

  // ---- column task ----
  const int k = static_cast<int>(blockIdx.x) - Pr;
  const int v = tid % kSmallColVecs;
  const int sl = tid / kSmallColVecs;
  const int c = k * kSmallColVecs + v;
  f2 acc[4], cmp[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[q] = f2_splat(0.f);
    cmp[q] = f2_splat(0.f);
  }
  if (c < NV) {
    constexpr int kB = 4;  // rows whose loads are in flight together
    for (int32_t r0 = sl; r0 < a.R; r0 += kB * kSmallSlices) {
      uint4 xb[kB], db[kB];
      float rb[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int32_t r = r0 + u * kSmallSlices;
        xb[u] = db[u] = make_uint4(0u, 0u, 0u, 0u);
        rb[u] = 0.f;
        if (r < a.R) {
          const int32_t t = r / a.map.nh;
          const int32_t hd = r - t * a.map.nh;
          xb[u] = *reinterpret_cast<const uint4*>(
              a.x + static_cast<int64_t>(t) * a.map.s_tok +
              static_cast<int64_t>(hd) * a.map.s_head + c * 8);
          db[u] = *reinterpret_cast<const uint4*>(a.dy + static_cast<size_t>(r) * H + c * 8);
          rb[u] = a.rstd[r];
        }
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if (r0 + u * kSmallSlices >= a.R) break;
        const float rs = rb[u];
        const float rs_hi = __uint_as_float(__float_as_uint(rs) & 0xffff0000u);
        const f2 rh2 = f2_splat(rs_hi);
        const f2 rl2 = f2_splat(__fsub_rn(rs, rs_hi));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const f2 dyx = f2_mul(bf2_to_f2(u4_get(db[u], q)), bf2_to_f2(u4_get(xb[u], q)));
          const f2 p = f2_mul(dyx, rh2);
          const f2 tt = f2_add(acc[q], p);
          const f2 e = f2_add(f2_sub(acc[q], tt), p);
          cmp[q] = f2_fma(dyx, rl2, f2_add(cmp[q], e));
          acc[q] = tt;
        }
      }
    }
  }
  float* sh = sm;                           // [kSmallSlices][kSmallCols] hi
  float* se = sm + kSmallSlices * kSmallCols;  // [kSmallSlices][kSmallCols] lo
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const f2 hi = f2_add(acc[q], cmp[q]);
    const f2 lo = f2_sub(cmp[q], f2_sub(hi, acc[q]));
    const int at = sl * kSmallCols + v * 8 + 2 * q;
    sh[at] = f2_lo(hi);
    sh[at + 1] = f2_hi(hi);
    se[at] = f2_lo(lo);
    se[at + 1] = f2_hi(lo);
  }
  __syncthreads();
#pragma unroll 1
  for (int stride = kSmallSlices / 2; stride > 0; stride >>= 1) {
    if (sl < stride) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int at = sl * kSmallCols + v * 8 + j;
        const int bt = (sl + stride) * kSmallCols + v * 8 + j;
        float err;
        const float S = two_sum_exact(sh[at], sh[bt], err);
        se[at] = __fadd_rn(__fadd_rn(se[at], se[bt]), err);
        sh[at] = S;
      }
    }
    __syncthreads();
  }
  if (sl == 0 && c < NV) {
    float out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) out[j] = __fadd_rn(sh[v * 8 + j], se[v * 8 + j]);
    float4* d = reinterpret_cast<float4*>(dw + c * 8);
    d[0] = make_float4(out[0], out[1], out[2], out[3]);
    d[1] = make_float4(out[4], out[5], out[6], out[7]);
  }
}

namespace {

template <int VPT>
const void* small_ptr_v(bool fp32w, bool dh) {
  if (fp32w)
    return dh ? reinterpret_cast<const void*>(&rmsn_bwd_small_kernel<VPT, true, true>)
              : reinterpret_cast<const void*>(&rmsn_bwd_small_kernel<VPT, true, false>);
  return dh ? reinterpret_cast<const void*>(&rmsn_bwd_small_kernel<VPT, false, true>)
            : reinterpret_cast<const void*>(&rmsn_bwd_small_kernel<VPT, false, false>);
}

}  // namespace


bool bwd_is_small(int64_t R) { return R > 0 && R <= kSmallMaxRows; }

// rstd of rows [0, a.R) for the backward that recomputes it on the one-launch path: one
// warp a row, the row's 16-byte vectors strided over the lanes, the sum of squares in FP32
// (BF16 squares are exact; the additions round), then the forward's correctly rounded
// 1/sqrt(sum/H + eps).
constexpr int kRstdRowsPerCta = 8;
__global__ void __launch_bounds__(32 * kRstdRowsPerCta)
    rmsn_rstd_rows_kernel(const BwdArgs a, float* __restrict__ rstd) {
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int H = a.map.H;
  const int NV = H >> 3;
  const int lane = threadIdx.x & 31;
  const int32_t row = static_cast<int32_t>(blockIdx.x) * kRstdRowsPerCta +
                      static_cast<int32_t>(threadIdx.x >> 5);
  if (row >= a.R) return;  // the whole warp
  const int32_t t = row / a.map.nh;
  const int32_t hd = row - t * a.map.nh;
  const __nv_bfloat16* xr = a.x + static_cast<int64_t>(t) * a.map.s_tok +
                            static_cast<int64_t>(hd) * a.map.s_head;
  f2 s0 = f2_splat(0.f), s1 = f2_splat(0.f);
  for (int c = lane; c < NV; c += 32) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c * 8);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const f2 x2 = bf2_to_f2(u4_get(v, q));
      if (q & 1)
        s1 = f2_fma(x2, x2, s1);
      else
        s0 = f2_fma(x2, x2, s0);
    }
  }
  const f2 sq = f2_add(s0, s1);
  const float ss = warp_allsum(f2_lo(sq) + f2_hi(sq));
  if (lane == 0)
    rstd[row] = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(H)), a.eps));
}

cudaError_t launch_rstd_rows(const BwdArgs& a, float* rstd, cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&rmsn_rstd_rows_kernel);
  BwdArgs copy = a;
  void* args[] = {&copy, &rstd};
  const unsigned grid = static_cast<unsigned>((a.R + kRstdRowsPerCta - 1) / kRstdRowsPerCta);
  return launch_pdl(fn, dim3(grid), dim3(32 * kRstdRowsPerCta), 0, st, args);
}

cudaError_t launch_bwd_small(const BwdArgs& a, float* dw, bool fp32w, cudaStream_t st) {
  const int NV = a.map.H / 8;
  const int vpt = (NV + kSmallThreads - 1) / kSmallThreads;  // 1..4 for H <= 8192
  const void* fn = vpt == 1 ? small_ptr_v<1>(fp32w, a.dh != nullptr)
                 : vpt == 2 ? small_ptr_v<2>(fp32w, a.dh != nullptr)
                 : vpt == 3 ? small_ptr_v<3>(fp32w, a.dh != nullptr)
                            : small_ptr_v<4>(fp32w, a.dh != nullptr);
  const int per = (NV + vpt - 1) / vpt;
  const int gt = per <= 32 ? 32 : (per + 31) / 32 * 32;
  const int groups = kSmallThreads / gt;
  int Pr = (a.R + groups - 1) / groups;
  const int Pc = (NV + kSmallColVecs - 1) / kSmallColVecs;
  BwdArgs copy = a;
  void* args[] = {&copy, &dw, &Pr};
  return launch_pdl(fn, dim3(static_cast<unsigned>(Pr + Pc)), dim3(kSmallThreads), 0, st,
                    args);
}

}  // namespace rmsn
