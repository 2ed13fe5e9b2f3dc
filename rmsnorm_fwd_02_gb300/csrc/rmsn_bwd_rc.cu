// rmsn_bwd_rc.cu -- the row-pass builds of the RMSNorm training backward that recompute
// rstd from the staged rows (rmsn_bwd_rows.cuh with kRc = true), in a translation unit of
// their own so that the builds compile in parallel.
#include "rmsn_bwd_rows.cuh"

namespace rmsn {

const void* bwd_rows_fn_rc(const Shape& s, bool fp32w, bool dh) {
  return pick_rows_kernel<true>(s, fp32w, dh);
}

}  // namespace rmsn
