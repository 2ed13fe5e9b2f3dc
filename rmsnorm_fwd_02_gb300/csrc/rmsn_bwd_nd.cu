// rmsn_bwd_nd.cu -- RMSNorm training backward for sm_103a, non-deterministic builds: the
// whole backward in one row-pass launch (rmsn_bwd_rows.cuh with kND = true), preceded by a
// one-CTA kernel that zeroes its control words and FP64 sums.
//
// flashinfer PR #8827 (description) leaves deterministic=False free to be faster, and the
// pages' non-deterministic routes are single kernels (PR #8848: "blocked FP32" dw sums in
// one kernel; PR #8899: the kb programs).  Here the mode buys two things the fixed
// partition cannot have: rows are handed out as the CTAs go (no CTA idles while another
// still has a queue of rows), and dw is finished by the last CTA without a second launch
// and a grid-wide drain in between.  dx is the deterministic build's, bit for bit.
#include "rmsn_bwd_rows.cuh"

namespace rmsn {

// Zeroes the row counter, the ticket counter and the H FP64 sums of one call.  It lets the
// row pass be scheduled at once (that grid still waits for this one to finish before it
// touches the workspace), and waits for the previous grid on the stream, which may be an
// earlier call still reading the same workspace.
__global__ void __launch_bounds__(256) rmsn_nd_prep_kernel(unsigned* ctl, double* acc, int H) {
  pdl_allow_next_grid();
  pdl_wait_prior_grid();
  if (threadIdx.x < kNdCtlBytes / sizeof(unsigned)) ctl[threadIdx.x] = 0u;
  double2* a2 = reinterpret_cast<double2*>(acc);  // 16-byte aligned: the workspace + 16
  for (int i = threadIdx.x; i < H / 2; i += blockDim.x) a2[i] = make_double2(0.0, 0.0);
}

const void* bwd_rows_fn_nd(const Shape& s, bool fp32w, bool dh) {
  return pick_rows_kernel<true, false>(s, fp32w, dh);
}

cudaError_t prepare_kernel(const void* fn, size_t smem);
int blocks_per_sm(const void* fn, int threads, size_t smem);
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       void** args);

int bwd_nd_blocks_per_sm(const Shape& s, bool fp32w, bool rc) {
  return blocks_per_sm(bwd_rows_fn(s, fp32w, s.tensors == 3, true, rc), s.threads, s.smem);
}

cudaError_t launch_bwd_nd(const BwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st) {
  const void* fn = bwd_rows_fn(s, fp32w, a.dh != nullptr, true, a.rstd == nullptr);
  cudaError_t e = prepare_kernel(fn, s.smem);
  if (e != cudaSuccess) return e;
  unsigned* ctl = a.ctl;
  double* acc = a.acc;
  int H = a.map.H;
  void* pargs[] = {&ctl, &acc, &H};
  e = launch_pdl(reinterpret_cast<const void*>(&rmsn_nd_prep_kernel), dim3(1), dim3(256), 0, st,
                 pargs);
  if (e != cudaSuccess) return e;
  BwdArgs copy = a;
  void* args[] = {&copy};
  return launch_pdl(fn, dim3(static_cast<unsigned>(a.P)), dim3(static_cast<unsigned>(s.threads)),
                    s.smem, st, args);
}

}  // namespace rmsn
