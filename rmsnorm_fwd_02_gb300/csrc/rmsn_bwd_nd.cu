// rmsn_bwd_nd.cu -- RMSNorm training backward for sm_103a, non-deterministic builds: the
// row pass of rmsn_bwd_rows.cuh with kND = true, whose CTAs take chunks of rows from an
// atomic counter as they go, followed by the fixed-order dw finish (which also clears the
// counter).
//
// flashinfer PR #8827 (description) leaves deterministic=False free to be faster.  What the
// mode buys here is the partition: with rows handed out as CTAs free up, no CTA idles
// while another still holds a queue of rows, and all CTAs stream through neighbouring rows
// together.  dx is the deterministic build's, bit for bit; dw's partials cover rows that
// vary from run to run, so its last bits may too.
#include "rmsn_bwd_rows.cuh"

namespace rmsn {

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
  BwdArgs copy = a;
  void* args[] = {&copy};
  return launch_pdl(fn, dim3(static_cast<unsigned>(a.P)), dim3(static_cast<unsigned>(s.threads)),
                    s.smem, st, args);
}

}  // namespace rmsn
