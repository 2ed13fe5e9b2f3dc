// ln_launch.h -- LayerNorm training: argument blocks, launch shapes and the shared-memory
// carve-up of the row kernels (host + device).
//
// The LayerNorm kernels stage rows exactly like the RMSNorm ones (rmsn_common.cuh: one
// producer warp, bulk asynchronous copies into an S-stage mbarrier ring, row groups of
// threads that own fixed 16-byte column vectors, split-phase rows); what differs is the
// per-row reduction (two quantities) and the backward's second column sum (db).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lnorm {

constexpr int kLnMaxH = 8192;
constexpr int kLnProducerThreads = 32;
constexpr int kLnRedBufs = 4;        // rotation of the per-row reduction buffers
constexpr int kLnMaxWarpsPerGroup = 16;

// Shape classes, each its own kernel build (and a CTA-pair build of each for widths past
// kLnMaxH) (launch bounds = consumers + producer warp):
//  kLnFwd       forward, up to 608 consumers, one CTA an SM (20 warps: 96 registers, which
//               the builds fit with w and b in shared memory)
//  kLnBwdMulti  backward with 1- or 2-vector threads, up to 480 consumers (128 registers)
//  kLnBwdWide   backward with 3-vector threads, up to 352 consumers (12 warps, three on a
//               scheduler partition: 168 registers), for rows past 480 2-vector threads;
//               the dw and db running sums and their compensations take 32 registers a
//               column vector
//  kLnFwdPair   forward of one CTA of a pair, up to 608 consumers (20 warps: 96 registers)
//  kLnBwdTm     backward with each thread's dw sums, their compensations and the db sums
//               in tensor memory (32 columns of its lane a column vector), up to 608
//               consumers (20 warps with the producer: 96 registers); single CTAs, and
//               (4 vectors a thread) one CTA of a pair
// (class 4 is not used: a register-resident 4-vector backward that the tensor-memory
// class replaced)
enum { kLnFwd = 0, kLnBwdMulti = 1, kLnBwdWide = 2, kLnFwdPair = 3, kLnBwdTm = 5 };
constexpr int ln_consumers(int cls) {
  return cls == kLnBwdWide ? 352
                           : ((cls == kLnBwdTm || cls == kLnFwd || cls == kLnFwdPair) ? 608 : 480);
}
// Tensor-memory columns a kLnBwdTm CTA of `cons_warps` consumer warps uses: 32 a column
// vector a thread (dw sums [0, 8), their compensations [8, 16), db sums [16, 24)), the
// warps sharing a lane quadrant side by side.
__host__ __device__ constexpr int ln_bwd_tm_cols(int cons_warps, int vpt) {
  return ((cons_warps + 3) / 4) * 32 * vpt;
}
constexpr int ln_max_threads(int cls) { return ln_consumers(cls) + kLnProducerThreads; }

// Floats per stage of a staged per-row FP32 array (mean, rstd): the stage's `rows` values
// start up to 3 floats into their first 16-byte block, and a slot stays whole blocks.
__host__ __device__ constexpr int ln_stat_stride(int rows) {
  return rows == 0 ? 0 : ((rows + 6) & ~3);
}

// Widths above kLnMaxH (up to kLnMaxHPair, multiples of 16) run as CTA pairs: a cluster of
// two CTAs per row chunk, each owning half of every row's columns (ln_common.cuh).
constexpr int kLnMaxHPair = 16384;
// Reduction slot floats per row group: two per warp, for the group's warps (single CTA) or
// for the warps of both CTAs of a pair.
constexpr int kLnSlotFloats = 32;
constexpr int kLnSlotFloatsPair = 64;
constexpr int kLnWtab = 32;  // entries per row of the forward's warp-merge table

// Byte offsets of a row kernel's shared memory (Hc = the columns this CTA owns: H, or H/2
// in a pair):
//   ring   [stages][tensors][groups][Hc] BF16 staged rows (offset 0)
//   full, empty   [stages] mbarriers
//   redb   [kLnRedBufs][red_groups] mbarriers of the per-row reductions
//   slots  [kLnRedBufs][red_groups][slot_floats] FP32: two partials per warp (2w, 2w+1)
//   stat   [stages][2][ln_stat_stride(stat_rows)] FP32 staged mean, rstd (backward)
//   head   [stages][head_rows] 16-byte heads of the staged rows (pair forward: the row's
//          first element, the shift both CTAs use)
//   wtab   [3][kLnWtab] FP32 per-warp counts, prefix counts and combine factors of the
//          forward's variance merge
//   w      the parameters in shared memory: the forward's w and b as FP32 (four planes of
//          float4: w columns 0-3, w 4-7, b 0-3, b 4-7 of every vector; 2*Hc floats), the
//          kLnBwdTm backward's w as given (BF16 or FP32; room for Hc floats)
//   abort  the CTA's abort flag of the bounded waits (word 0); word 2: the tensor-memory
//          address of the kLnBwdTm builds
struct LnSmem {
  size_t full, empty, redb, slots, stat, head, wtab, w, abort_flag, total;
};

__host__ __device__ inline LnSmem ln_smem_layout(int stages, int tensors, int groups, int Hc,
                                                 int red_groups, int stat_rows,
                                                 int slot_floats, int head_rows,
                                                 int w_floats = 0) {
  LnSmem L;
  size_t off = static_cast<size_t>(stages) * tensors * groups * Hc * 2;  // multiple of 16
  L.full = off;
  off += 8 * static_cast<size_t>(stages);
  L.empty = off;
  off += 8 * static_cast<size_t>(stages);
  L.redb = off;
  off += 8 * kLnRedBufs * static_cast<size_t>(red_groups);
  off = (off + 127) & ~static_cast<size_t>(127);
  L.slots = off;
  off += 4 * kLnRedBufs * static_cast<size_t>(slot_floats) * red_groups;
  L.stat = off;  // 128-byte aligned
  off += 4 * static_cast<size_t>(stages) * 2 * ln_stat_stride(stat_rows);
  L.head = off;  // 16-byte aligned
  off += 16 * static_cast<size_t>(stages) * head_rows;
  L.wtab = off;  // 16-byte aligned
  off += 4 * 3 * kLnWtab;
  L.w = off;  // 16-byte aligned
  off += 4 * static_cast<size_t>(w_floats);
  L.abort_flag = off;
  off += 16;
  L.total = off;
  return L;
}

struct LnShape {
  int vpt;      // 16-byte column vectors per consumer thread
  int ntg;      // threads per row group: 8, 16 or a multiple of 32
  int groups;   // row groups per CTA = rows per stage
  int stages;   // ring depth
  int tensors;  // BF16 tensors staged per row (1 forward, 2 backward)
  int threads;  // groups * ntg + producer warp
  size_t smem;  // dynamic shared memory bytes
  int cls;      // kLnFwd, kLnBwdMulti, kLnBwdWide, kLnFwdPair or kLnBwdTm
  int pair;     // 1: a CTA pair per row chunk, each CTA owning half the columns
};

struct LnFwdArgs {
  const __nv_bfloat16* x;  // [R, H]
  const void* w;           // [H]
  const void* b;           // [H], same dtype as w
  __nv_bfloat16* y;        // [R, H]
  float* mean;             // [R]
  float* rstd;             // [R]
  int32_t R, H;
  float eps;
  int32_t groups, ntg, stages, P;
  unsigned* err;
};

struct LnBwdArgs {
  const __nv_bfloat16* x;   // [R, H]
  const __nv_bfloat16* dy;  // [R, H]
  const float* mean;        // [R]
  const float* rstd;        // [R]
  const void* w;            // [H]
  __nv_bfloat16* dx;        // [R, H]
  float* part;              // [P][2][2H]: per CTA, (hi, lo) rows over dw's H then db's H
  int32_t R, H;
  int32_t groups, ntg, stages, P;
  unsigned* err;
};

LnShape ln_fwd_shape(int H);
LnShape ln_bwd_shape(int H);

// Shared memory of a shape (host and kernels agree through ln_smem_layout).
__host__ __device__ inline LnSmem ln_shape_layout(int stages, int tensors, int groups, int H,
                                                  int ntg, bool pair, bool bwd_w_smem = false) {
  const int Hc = pair ? H / 2 : H;
  const int w_floats = tensors == 1 ? 2 * Hc : (bwd_w_smem ? Hc : 0);
  return ln_smem_layout(stages, tensors, groups, Hc, ntg >= 32 ? groups : 0,
                        tensors == 2 ? groups : 0, pair ? kLnSlotFloatsPair : kLnSlotFloats,
                        pair && tensors == 1 ? groups : 0, w_floats);
}

cudaError_t ln_launch_fwd(const LnFwdArgs& a, const LnShape& s, bool fp32w, cudaStream_t st);
cudaError_t ln_launch_bwd_rows(const LnBwdArgs& a, const LnShape& s, bool fp32w,
                               cudaStream_t st);
cudaError_t ln_launch_finish(const float* part, float* dw, float* db, int P, int H,
                             cudaStream_t st);
// Launches `pairs` clusters of two CTAs (grid 2 * pairs) of a pair build.
cudaError_t ln_launch_pair(const void* fn, unsigned pairs, unsigned threads, size_t smem,
                           cudaStream_t st, void** args);
int ln_fwd_blocks_per_sm(const LnShape& s, bool fp32w);
int ln_bwd_blocks_per_sm(const LnShape& s, bool fp32w);

}  // namespace lnorm
