// rmsn_launch.h -- kernel argument blocks and launcher entry points (host + device).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

constexpr int kMaxH = 8192;
constexpr int kProducerThreads = 32;       // one warp; lane 0 issues the bulk copies
constexpr int kMaxConsumerThreads = 512;   // G * NTg
constexpr int kMaxThreads = kMaxConsumerThreads + kProducerThreads;
constexpr int kFinishCols = 32;            // dw columns per finishing CTA
constexpr int kFinishSlices = 8;           // partition slices per finishing CTA

// Launch shape of a row kernel, a function of H (and of the mode for P).
struct Shape {
  int vpt;       // 16-byte column vectors per consumer thread (1 or 2)
  int ntg;       // threads per row group (a multiple of 32)
  int groups;    // row groups per CTA = rows per stage
  int stages;    // depth of the shared-memory ring
  int tensors;   // BF16 tensors staged per row
  int threads;   // groups * ntg + producer warp
  size_t smem;   // dynamic shared memory bytes
};

struct RowMapArgs {
  int32_t nh;
  int32_t H;
  int64_t s_tok;
  int64_t s_head;
};

struct FwdArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* res;   // nullable
  const void* w;
  __nv_bfloat16* y;
  __nv_bfloat16* h;           // nullable iff res is null
  float* rstd;
  RowMapArgs map;
  int32_t R;                  // normalized rows = T * nh
  int32_t contig;             // input row r starts at element r * H
  float eps;
  int32_t groups, ntg, stages, P;
  unsigned* err;              // device error word
};

struct BwdArgs {
  const __nv_bfloat16* x;     // forward's normalized input, strided
  const __nv_bfloat16* dy;    // contiguous
  const __nv_bfloat16* dh;    // contiguous, nullable
  const float* rstd;
  const void* w;
  __nv_bfloat16* dx;          // contiguous
  float* part;                // [P][2][H]: compensated dw partial per CTA (hi row, lo row)
  RowMapArgs map;
  int32_t R;
  int32_t contig;
  int32_t groups, ntg, stages, P;
  unsigned* err;
};

// Shape of the forward / backward row kernels for width H.
Shape fwd_shape(int H, bool residual);
Shape bwd_shape(int H, bool with_dh);

// Launchers: return the CUDA launch status.  `pdl` opts the launch into programmatic
// dependent launch (overlap with the previous kernel on the stream).
cudaError_t launch_fwd(const FwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st);
cudaError_t launch_bwd_rows(const BwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st);
cudaError_t launch_dw_finish(const float* part, float* dw, int P, int H, cudaStream_t st);

// CTAs per SM the backward row kernel is built to keep resident (its launch bounds'
// minimum), a compile-time property: 2 for one-vector threads, else 1.
constexpr int bwd_design_blocks_per_sm(int vpt) { return vpt == 1 ? 2 : 1; }

// Resident CTAs per SM of the chosen row kernel (cached per device).
int fwd_blocks_per_sm(const Shape& s, bool fp32w);
int bwd_blocks_per_sm(const Shape& s, bool fp32w);

}  // namespace rmsn
