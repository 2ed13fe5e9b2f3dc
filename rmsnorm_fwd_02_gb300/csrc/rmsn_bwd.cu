// rmsn_bwd.cu -- RMSNorm training backward for sm_103a: the row pass (rmsn_bwd_rows.cuh;
// its builds that read rstd -- those that recompute it are in rmsn_bwd_rc.cu), each CTA
// writing its compensated dw partial to the workspace, and the fixed-order dw finish.
//
// One row-pass program serves both modes.  deterministic=1: CTA k owns a fixed chunk of
// rows, a function of (R, P) only.  deterministic=0 (flashinfer PR #8827, description:
// free to be faster): each CTA owns a fixed prefix and the last rows are handed out from a
// counter in the workspace as CTAs free up, so no CTA idles while another still holds a
// queue of rows; dw's partials then cover rows that vary from run to run, so its last bits
// may too (with fewer than eight ring depths of rows a CTA, the deterministic chunks).  dx
// never depends on the partition: it is bit-identical across the modes.
#include "rmsn_bwd_rows.cuh"

namespace rmsn {

// dw[col] = sum over k = 0..P-1 of (hi_k + lo_k), in a fixed order: slice i of the
// kFinishSlices slices takes k in [i*P/slices, (i+1)*P/slices) in increasing k, then the
// slice sums are combined by a pairwise tree in slice order (i with i + stride, stride
// halving).  TwoSum carries the error terms throughout.  Each thread walks only ~P/32
// partials, so the kernel is a short tail.  Two builds add them the same way and differ
// only in how the loads are batched: kOneTrip loads up to five (hi, lo) pairs at once, so
// a slice of P <= 160 partials takes one round trip to L2 (64 registers: one 1024-thread
// CTA an SM, taken when the grid fits one wave), the other four at a time and the rest one
// by one (32 registers: two CTAs an SM).
template <bool kOneTrip>
__global__ void __launch_bounds__(kFinishCols* kFinishSlices)
    rmsn_dw_finish_kernel(const float* __restrict__ part, float* __restrict__ dw, int P, int H,
                          unsigned* ctl) {
  __shared__ float sh[kFinishSlices][kFinishCols];
  __shared__ float se[kFinishSlices][kFinishCols];
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  // the row pass that used the non-deterministic pool is complete: clear its words, so
  // that a replay of this call (same tag) finds the pool closed until its CTA 0 opens it
  if (ctl != nullptr && blockIdx.x == 0 && threadIdx.x < 2) ctl[threadIdx.x] = 0u;
  const int cl = threadIdx.x % kFinishCols;
  const int sl = threadIdx.x / kFinishCols;
  const int col = blockIdx.x * kFinishCols + cl;
  float s = 0.f, e = 0.f;
  if (col < H) {
    const int ka = (sl * P) / kFinishSlices;
    const int kb = ((sl + 1) * P) / kFinishSlices;
    const float* p = part + static_cast<size_t>(ka) * 2 * H + col;
    if constexpr (kOneTrip) {
      for (int kk = ka; kk < kb; kk += 5, p += static_cast<size_t>(10) * H) {
        const int n = kb - kk;
        float hi[5], lo[5];
#pragma unroll
        for (int u = 0; u < 5; ++u) {
          if (u < n) {
            hi[u] = p[static_cast<size_t>(2 * u) * H];
            lo[u] = p[static_cast<size_t>(2 * u + 1) * H];
          }
        }
#pragma unroll
        for (int u = 0; u < 5; ++u) {
          if (u < n) {
            float err;
            s = two_sum(s, hi[u], err);
            e = __fadd_rn(e, __fadd_rn(err, lo[u]));
          }
        }
      }
    } else {
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

const void* bwd_rows_fn_rs(const Shape& s, bool fp32w, bool dh) {
  return pick_rows_kernel<false>(s, fp32w, dh);
}

const void* bwd_rows_fn(const Shape& s, bool fp32w, bool dh, bool rc) {
  return rc ? bwd_rows_fn_rc(s, fp32w, dh) : bwd_rows_fn_rs(s, fp32w, dh);
}

int bwd_blocks_per_sm(const Shape& s, bool fp32w, bool rc) {
  return blocks_per_sm(bwd_rows_fn(s, fp32w, s.tensors == 3, rc), s.threads, s.smem);
}

cudaError_t launch_bwd_rows(const BwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st) {
  const void* fn = bwd_rows_fn(s, fp32w, a.dh != nullptr, a.rstd == nullptr);
  cudaError_t e = prepare_kernel(fn, s.smem);
  if (e != cudaSuccess) return e;
  BwdArgs copy = a;
  void* args[] = {&copy};
  return launch_pdl(fn, dim3(static_cast<unsigned>(a.P)), dim3(static_cast<unsigned>(s.threads)),
                    s.smem, st, args);
}

cudaError_t launch_dw_finish(const float* part, float* dw, int P, int H, unsigned* ctl,
                             int sms, cudaStream_t st) {
  void* args[] = {&part, &dw, &P, &H, &ctl};
  const unsigned grid = static_cast<unsigned>((H + kFinishCols - 1) / kFinishCols);
  const void* fn = grid <= static_cast<unsigned>(sms)
                       ? reinterpret_cast<const void*>(&rmsn_dw_finish_kernel<true>)
                       : reinterpret_cast<const void*>(&rmsn_dw_finish_kernel<false>);
  return launch_pdl(fn, dim3(grid), dim3(kFinishCols * kFinishSlices), 0, st, args);
}

}  // namespace rmsn
