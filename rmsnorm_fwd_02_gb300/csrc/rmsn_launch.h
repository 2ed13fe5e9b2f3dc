// rmsn_launch.h -- kernel argument blocks and launcher entry points (host + device).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

constexpr int kMaxH = 8192;
constexpr int kProducerThreads = 32;       // one warp; lane 0 issues the bulk copies
constexpr int kMaxConsumerThreads = 512;   // G * NTg
constexpr int kFinishCols = 32;            // dw columns per finishing CTA
constexpr int kFinishSlices = 32;          // partition slices per finishing CTA

// Shared-memory carve-up of a row kernel (byte offsets), used by the kernels and by the
// host's size computation alike.
//   ring   [stages][tensors][groups][H] BF16 staged rows
//   full, empty   [stages] mbarriers (staged bytes landed / stage released)
//   redb   [kRedBufs][groups] mbarriers: a row's per-warp reduction partials are written
//   slots  [kRedBufs][groups][32] FP32 per-warp reduction partials
//   rs     [stages][rs_stride(rs_rows)] FP32: the staged rows' rstd (backward; forward:
//          none), from the 16-byte block holding the stage's first row onwards
//   w      [w_floats] FP32 weight, for builds that keep it in shared memory
//   abort  CTA abort flag of the bounded waits (word 0); word 2: the tensor-memory
//          address of the backward builds that keep their dw sums there
//   srow   [srow_stages] int32: the first and end row of each staged chunk (builds
//          whose producer decides its chunks as it goes: 2 per stage; others: none)
//
// Row j's reduction uses buffer j % kRedBufs.  A warp writes buffer j in phase A(j) after
// finishing B(j-2), which needed every warp's A(j-2), which each warp issues after its
// own B(j-4): so every reader of buffer j-4 is done, and four buffers never race.  The
// same ordering keeps each redb barrier within one phase of its waiters.
constexpr int kRedBufs = 4;
struct SmemLayout {
  size_t full, empty, redb, slots, rs, w, abort_flag, srow, total;
};

// Floats per stage of the staged rstd: the stage's `rows` values start up to 3 floats
// into their first 16-byte block, and a stage slot stays a whole number of blocks.
__host__ __device__ constexpr int rs_stride(int rows) { return rows == 0 ? 0 : ((rows + 6) & ~3); }

// `red_groups` is the number of row groups that reduce through shared memory: all of them
// when a group spans whole warps, none when groups are sub-warp (shuffles only).
// `rs_rows` is the number of rstd values staged with each stage (the backward's groups).
__host__ __device__ inline SmemLayout smem_layout(int stages, int tensors, int groups, int H,
                                                  int red_groups, int rs_rows,
                                                  int w_floats = 0, int srow_stages = 0) {
  SmemLayout L;
  size_t off = static_cast<size_t>(stages) * tensors * groups * H * 2;  // multiple of 16
  L.full = off;
  off += 8 * static_cast<size_t>(stages);
  L.empty = off;
  off += 8 * static_cast<size_t>(stages);
  L.redb = off;
  off += 8 * kRedBufs * static_cast<size_t>(red_groups);
  off = (off + 127) & ~static_cast<size_t>(127);
  L.slots = off;
  off += 4 * kRedBufs * 32 * static_cast<size_t>(red_groups);
  L.rs = off;  // 128-byte aligned
  off += 4 * static_cast<size_t>(stages) * rs_stride(rs_rows);
  L.w = off;   // 16-byte aligned
  off += 4 * static_cast<size_t>(w_floats);
  L.abort_flag = off;
  off += 16;
  L.srow = off;
  off += 4 * ((static_cast<size_t>(srow_stages) + 3) & ~static_cast<size_t>(3));
  L.total = off;
  return L;
}

// Launch shape of a row kernel, a function of H (and of the mode for P).
struct Shape {
  int vpt;       // 16-byte column vectors per consumer thread (1..4)
  int ntg;       // threads per row group: 8 or 16 (sub-warp) or a multiple of 32
  int groups;    // row groups per CTA = rows per stage
  int stages;    // depth of the shared-memory ring
  int tensors;   // BF16 tensors staged per row
  int threads;   // groups * ntg + producer warp
  size_t smem;   // dynamic shared memory bytes
  int cls;       // shape class: kFwdPair / kFwdSolo, or kBwdNarrow / kBwdMulti / kBwdWide /
                 // kBwdTm
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
  // non-deterministic builds: ctl[0] the tag of the call that opened the tail-row pool,
  // ctl[1] the next pool row; tag is nonzero and differs from call to call (a CUDA graph
  // replays its call's tag, and the finish clears ctl[0] between calls)
  unsigned* ctl;
  uint32_t tag;
  // rstd == nullptr: the row pass recomputes rstd (eps as in the forward) and writes it to
  // rstd_out when that is not null
  float eps;
  float* rstd_out;
  RowMapArgs map;
  int32_t R;
  int32_t contig;
  int32_t groups, ntg, stages, P;
  unsigned* err;
};

// Shape of the forward / backward row kernels for width H.
Shape fwd_shape(int H, bool residual);
Shape bwd_shape(int H, bool with_dh);  // both modes

// Launchers: return the CUDA launch status.  `pdl` opts the launch into programmatic
// dependent launch (overlap with the previous kernel on the stream).
cudaError_t launch_fwd(const FwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st);
// The row-pass kernel build for a shape (one program for both modes), with rstd given or
// recomputed (rc): rmsn_bwd.cu and rmsn_bwd_rc.cu.
const void* bwd_rows_fn(const Shape& s, bool fp32w, bool dh, bool rc);
const void* bwd_rows_fn_rs(const Shape& s, bool fp32w, bool dh);
const void* bwd_rows_fn_rc(const Shape& s, bool fp32w, bool dh);
int bwd_blocks_per_sm(const Shape& s, bool fp32w, bool rc);

// The row pass, either mode: a.ctl null (deterministic: fixed chunks) or the
// non-deterministic pool's words.
cudaError_t launch_bwd_rows(const BwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st);
// ctl: the non-deterministic pool words to clear once the partials are summed, or null;
// sms: the GPU's SM count (the finish build that takes a whole SM a CTA runs only where
// its grid fits one wave).
cudaError_t launch_dw_finish(const float* part, float* dw, int P, int H, unsigned* ctl,
                             int sms, cudaStream_t st);

// The non-deterministic workspace starts with the pool's two words (a 16-byte slot),
// followed by the P partials; the fixed-order finish adds the partials and clears the
// words.  They need no initial value: the pool is open to a call only once its CTA 0 has
// published the call's tag there.
constexpr size_t kNdCtlBytes = 16;

// Small inputs (rmsn_small.cu): the whole backward in one launch of row tasks (dx) and
// column tasks (dw over every row in a fixed order), no workspace, for R <= kSmallMaxRows.
constexpr int kSmallThreads = 256;
constexpr int kSmallColVecs = 4;                              // column vectors a column task
constexpr int kSmallSlices = kSmallThreads / kSmallColVecs;   // row slices a column task
constexpr int64_t kSmallMaxRows = 256;
bool bwd_is_small(int64_t R);
cudaError_t launch_bwd_small(const BwdArgs& a, float* dw, bool fp32w, cudaStream_t st);
// rstd of rows [0, R) into `rstd` (one warp a row, the forward's formula), for the small
// path of the backward that recomputes rstd.
cudaError_t launch_rstd_rows(const BwdArgs& a, float* rstd, cudaStream_t st);

// Backward shape classes, each its own kernel build:
//  kBwdNarrow  up to 256 consumers, two CTAs an SM: one-vector lanes (H = 8)
//  kBwdMulti   2- to 4-vector threads in row groups of 8, 16 or 32..240 threads, as many
//              groups as fit in 480 consumers (at most 16 whole-warp groups), one CTA an
//              SM: several rows in flight per CTA
//              (4-vector threads keep the weight in shared memory, not registers).  With
//              the producer that is 16 warps, four a scheduler partition, which leaves
//              128 registers a thread (17 warps would put five warps on one partition
//              and cap every thread at 96, too few for the dw state without spills)
//  kBwdWide    one row group of more than 240 threads (2-vector, H up to 6144) or
//              4-vector threads (H above 6144), one CTA an SM
//  kBwdTm      the multi-group class with each thread's dw sums and compensation in
//              tensor memory instead of registers, and the weight in shared memory: up
//              to 608 consumers (20 warps with the producer, 96 registers a thread), so
//              more rows in flight where the multi class's registers run out
enum { kBwdNarrow = 0, kBwdMulti = 1, kBwdWide = 2, kBwdTm = 3 };
constexpr int kMultiConsumers = 480;
constexpr int kTmConsumers = 608;

// Backward builds that keep the weight in shared memory (FP32, H floats) instead of
// registers: 4-vector threads of the multi-group class, and the tensor-memory class.
__host__ __device__ constexpr bool bwd_w_in_smem(int cls, int vpt) {
  return cls == kBwdTm || (cls == kBwdMulti && vpt == 4);
}

// Tensor-memory columns a kBwdTm CTA of `cons_warps` consumer warps allocates: per thread
// 16 columns a vector (8 sums, then 8 compensation terms), the warps that share a lane
// quadrant side by side.
__host__ __device__ constexpr int bwd_tm_cols(int cons_warps, int vpt) {
  return ((cons_warps + 3) / 4) * 16 * vpt;
}

// CTAs per SM the backward row kernel is built to keep resident (its launch bounds'
// minimum), a compile-time property of the shape class.
constexpr int bwd_design_blocks_per_sm(int cls) { return cls == kBwdNarrow ? 2 : 1; }

// Threads a backward CTA of the class may have (its launch bounds' maximum).
constexpr int bwd_max_threads(int cls, int vpt) {
  return kProducerThreads +
         (cls == kBwdMulti ? kMultiConsumers
                           : (cls == kBwdTm ? kTmConsumers
                                            : (cls == kBwdWide && vpt == 2 ? 384 : 256)));
}

// Forward shape classes:
//  kFwdPair  up to 256 consumers + the producer warp, two CTAs an SM: sub-warp groups
//            and rows of at most 32-thread groups
//  kFwdSolo  one CTA an SM, row groups of 64 or more threads (or one-warp rows of 6
//            vectors a thread), as many as fit (at most 16): 512 consumers + the producer
//            warp for 2-4 vectors a thread (17 warps, at most 96 registers, which these
//            builds fit), 480 for 6 (16 warps, 128 registers)
// Two CTAs an SM split its bandwidth unevenly (one of the pair finishes its equal share
// first and the other then runs alone); one CTA holding the same number of rows in
// flight avoids that, where a row group is large enough to keep the warps busy.
enum { kFwdPair = 0, kFwdSolo = 1 };
constexpr int fwd_solo_consumers(int vpt) { return vpt == 6 ? 480 : 512; }
constexpr int fwd_design_blocks_per_sm(int cls) { return cls == kFwdPair ? 2 : 1; }
constexpr int fwd_max_threads(int cls, int vpt) {
  return kProducerThreads + (cls == kFwdPair ? 256 : fwd_solo_consumers(vpt));
}

// Resident CTAs per SM of the chosen row kernel (cached per device).
int fwd_blocks_per_sm(const Shape& s, bool fp32w);

}  // namespace rmsn
