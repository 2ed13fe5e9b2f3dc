// rmsn_fwd.cu -- RMSNorm training forward for sm_103a.
//
// Computes, per normalized row (flashinfer PR #8827, description; Measurement workload
// line: eps 1e-6, y and h_new BF16, rstd FP32):
//   [residual form]  h = BF16(x_in + residual)        (written; the norm is taken of h)
//   rstd = 1 / sqrt(sum_j x_j^2 / H + eps)             (FP32)
//   y_j  = BF16((x_j * rstd) * w_j)                    (round to nearest even)
//
// HBM-bound: 4 bytes per element (8 in the residual form) for ~3 flops.  Rows are staged
// into shared memory by bulk asynchronous copies (one producer thread, S-stage mbarrier
// ring) and consumed by row groups whose threads own fixed 16-byte column vectors, so
// every global access is a 16-byte coalesced vector and the weight stays in registers.
//
// Split-phase rows: phase A of row j reads the row and forms each thread's partial sum
// of squares; phase B of row j-1 re-reads row j-1 from shared memory into registers,
// releases the stage, waits for row j-1's reduction (published one iteration earlier, so
// normally complete) and writes y; then row j's warp partials are published.  No warp
// ever blocks on the row it is still reducing.
//
// Precision: the sum of squares is accumulated in FP32 (BF16 squares are exact in FP32,
// so only the additions round); the reciprocal square root is the correctly rounded
// __frsqrt_rn, which keeps rstd within 1e-6 relative of the FP64 value.  Arithmetic runs
// on packed FP32 pairs (f32x2).
#include "rmsn_common.cuh"
#include "rmsn_launch.h"

namespace rmsn {

// h = BF16(x_in + residual) for one 16-byte vector.  The FP32 sum of two BF16 values is
// exact unless their exponents differ by more than 16, and then the smaller one is far
// below half a BF16 ulp of the larger: either way the rounding gives BF16_RNE of the
// exact sum.
__device__ __forceinline__ uint4 residual_sum8(const uint4& u, const uint4& q) {
  uint4 r;
  r.x = f2_to_bf2(f2_add(bf2_to_f2(u.x), bf2_to_f2(q.x)));
  r.y = f2_to_bf2(f2_add(bf2_to_f2(u.y), bf2_to_f2(q.y)));
  r.z = f2_to_bf2(f2_add(bf2_to_f2(u.z), bf2_to_f2(q.z)));
  r.w = f2_to_bf2(f2_add(bf2_to_f2(u.w), bf2_to_f2(q.w)));
  return r;
}

// Launch bounds per shape class (rmsn_launch.h): kFwdPair, at most 256 consumers (G*NTg)
// + the producer warp, two CTAs an SM; kFwdSolo, at most 512 consumers (480 with 6
// vectors a thread) + the producer warp, one CTA an SM.
// Narrow rows use sub-warp groups of 8 or 16 lanes (several rows a warp, reduced by
// shuffles alone).
template <int VPT, int kCls, bool kFp32W, bool kRes>
__global__ void __launch_bounds__(fwd_max_threads(kCls, VPT), fwd_design_blocks_per_sm(kCls))
    rmsn_fwd_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NT = kRes ? 2 : 1;
  const int H = a.map.H;
  const int NV = H >> 3;
  const int G = a.groups, NTg = a.ntg, S = a.stages;
  const int NW = NTg >> 5;
  const size_t stage_elems = static_cast<size_t>(NT) * G * H;
  const bool red_smem = NTg >= 32;  // else sub-warp groups: shuffles only
  const SmemLayout L = smem_layout(S, NT, G, H, red_smem ? G : 0, 0);

  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  uint64_t* redb = reinterpret_cast<uint64_t*>(smem + L.redb);  // [kRedBufs][G]
  float* slots = reinterpret_cast<float*>(smem + L.slots);       // [kRedBufs][G][32]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

  const int tid = threadIdx.x;
  const int ncons = G * NTg;
  const int32_t k = blockIdx.x;
  const int32_t r0 = static_cast<int32_t>((static_cast<int64_t>(k) * a.R) / a.P);
  const int32_t r1 = static_cast<int32_t>((static_cast<int64_t>(k + 1) * a.R) / a.P);
  const int32_t nstage = (r1 - r0 + G - 1) / G;

  if (tid >= ncons) {  // the producer warp
    init_row_barriers_warp(full, empty, S, static_cast<uint32_t>(G * NTg / 32), redb,
                           red_smem ? kRedBufs * G : 0, static_cast<uint32_t>(NW), tid - ncons);
    if (tid == ncons) *abort_flag = 0;
  }
  __syncthreads();
  // Inputs may come from the kernel before us on the stream: wait for it before any
  // global read, then let the next kernel start its prologue.
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  if (tid >= ncons) {  // ---- producer warp ----
    if (tid == ncons) {
      const uint64_t pol = l2_evict_first_policy();
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
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rb - ra) * H * 2u * NT);
        __nv_bfloat16* dst = ring + s * stage_elems;
        if (a.contig) {
          copy_rows_contig(dst, a.x, H, ra, rb, &full[s], pol);
          if constexpr (kRes) copy_rows_contig(dst + G * H, a.res, H, ra, rb, &full[s], pol);
        } else {
          copy_rows(dst, a.x, m, ra, rb, &full[s], pol);
          if constexpr (kRes) copy_rows(dst + G * H, a.res, m, ra, rb, &full[s], pol);
        }
      }
      mbar_drain(full, S, j);
    }
    return;
  }

  // ---- consumers: group g, thread lt owns column vectors c = lt + v*NTg ----
  const int g = tid / NTg;
  const int lt = tid - g * NTg;
  const int wg = lt >> 5, lane = tid & 31;
  f2 wv[VPT][4];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = lt + v * NTg;
    if (c < NV) load_w8_pairs<kFp32W>(a.w, c, wv[v]);
  }
  const float hf = static_cast<float>(H);  // exact for H < 2^24
  // Rows of this warp's first group: every lane of a warp runs the same iterations (the
  // shuffles need them all); groups past the chunk's end skip the row work.
  const int g0 = red_smem ? g : (tid & ~31) / NTg;
  const int32_t ng = (r1 - r0 > g0) ? (r1 - r0 - g0 + G - 1) / G : 0;

  float ss_carry = 0.f;  // sub-warp groups: row j-1's sum of squares
  int s_cur = 0, s_prev = 0;  // slot and parity of stage j, slot of stage j-1 (increments,
  uint32_t ph = 0;            // no division by the runtime ring depth)
  for (int32_t j = 0; j <= ng; ++j) {
    float part = 0.f;
    // ---- phase A, row j: this thread's partial sum of squares (and h, residual form) ----
    if (j < ng) {
      const int32_t row = r0 + j * G + g;
      const int s = s_cur;
      mbar_wait_bounded(&full[s], ph, abort_flag, a.err, kErrConsumerWait);
      const __nv_bfloat16* xs = ring + s * stage_elems + static_cast<size_t>(g) * H;
      f2 ss0 = f2_splat(0.f), ss1 = f2_splat(0.f);  // two chains, fixed combine order
      if (row < r1) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
            uint4 u = lds128(xs + c * 8);
            if constexpr (kRes) {
              u = residual_sum8(u, lds128(xs + static_cast<size_t>(G) * H + c * 8));
              stg128(a.h + static_cast<size_t>(row) * H + c * 8, u);
            }
            // x^2 + ss per element straight from the BF16 words (the square is exact, so
            // this rounds exactly as converting first and using an FP32 fma would)
            ss0 = bf2_sq_acc(u.x, ss0);
            ss1 = bf2_sq_acc(u.y, ss1);
            ss0 = bf2_sq_acc(u.z, ss0);
            ss1 = bf2_sq_acc(u.w, ss1);
          }
        }
      }
      const f2 sp = f2_add(ss0, ss1);
      part = f2_lo(sp) + f2_hi(sp);
    }
    // ---- phase B, row j-1: rstd, y ----
    // Its staged vectors go to registers first and the stage is released at once; then
    // the row's reduction result is awaited (normally long complete), and row j's warp
    // reduction runs inside B's arithmetic, where its shuffle chain overlaps B's math.
    float red_j = 0.f;
    if (j >= 1) {
      const int32_t jj = j - 1;
      const int32_t row = r0 + jj * G + g;
      const int s = s_prev;
      const bool valid = row < r1;
      const __nv_bfloat16* xs = ring + s * stage_elems + static_cast<size_t>(g) * H;
      uint4 hv[VPT];
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = lt + v * NTg;
        hv[v] = make_uint4(0u, 0u, 0u, 0u);
        if (valid && c < NV) {
          hv[v] = lds128(xs + c * 8);
          if constexpr (kRes)
            hv[v] = residual_sum8(hv[v], lds128(xs + static_cast<size_t>(G) * H + c * 8));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp has its vectors of the stage
      float ss = ss_carry;
      if (red_smem) {
        const int rb = (jj % kRedBufs) * G + g;
        mbar_wait_bounded(&redb[rb], static_cast<uint32_t>(jj / kRedBufs) & 1u, abort_flag,
                          a.err, kErrConsumerWait);
        ss = slot_sum(slots + rb * 32, NW);
      }
      if (j < ng) red_j = red_smem ? warp_allsum(part) : subwarp_allsum(part, NTg);
      if (valid) {
        const float rs = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, hf), a.eps));
        const f2 rs2 = f2_splat(rs);
        const size_t out_row = static_cast<size_t>(row) * H;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
            uint4 o;
            o.x = f2_to_bf2(f2_mul(f2_mul(bf2_to_f2(hv[v].x), rs2), wv[v][0]));
            o.y = f2_to_bf2(f2_mul(f2_mul(bf2_to_f2(hv[v].y), rs2), wv[v][1]));
            o.z = f2_to_bf2(f2_mul(f2_mul(bf2_to_f2(hv[v].z), rs2), wv[v][2]));
            o.w = f2_to_bf2(f2_mul(f2_mul(bf2_to_f2(hv[v].w), rs2), wv[v][3]));
            stg128(a.y + out_row + c * 8, o);
          }
        }
        if (lt == 0) a.rstd[row] = rs;
      }
    } else if (j < ng) {
      red_j = red_smem ? warp_allsum(part) : subwarp_allsum(part, NTg);
    }
    // ---- publish row j's reduction ----
    if (j < ng && red_smem && lane == 0) {
      slots[((j % kRedBufs) * G + g) * 32 + wg] = red_j;
      mbar_arrive(&redb[(j % kRedBufs) * G + g]);
    }
    ss_carry = red_j;
    s_prev = s_cur;
    if (++s_cur == S) {
      s_cur = 0;
      ph ^= 1u;
    }
  }
}

template <int VPT, int kCls, bool kFp32W, bool kRes>
static const void* fwd_kernel_ptr() {
  return reinterpret_cast<const void*>(&rmsn_fwd_kernel<VPT, kCls, kFp32W, kRes>);
}

template <int VPT, int kCls>
static const void* pick_fwd_v(bool fp32w, bool res) {
  if (fp32w)
    return res ? fwd_kernel_ptr<VPT, kCls, true, true>() : fwd_kernel_ptr<VPT, kCls, true, false>();
  return res ? fwd_kernel_ptr<VPT, kCls, false, true>() : fwd_kernel_ptr<VPT, kCls, false, false>();
}

// kFwdSolo is built for 2, 3, 4 and 6 vectors a thread, kFwdPair for 1 to 4.
static const void* pick_fwd(const Shape& s, bool fp32w, bool res) {
  if (s.cls == kFwdSolo) {
    switch (s.vpt) {
      case 2: return pick_fwd_v<2, kFwdSolo>(fp32w, res);
      case 3: return pick_fwd_v<3, kFwdSolo>(fp32w, res);
      case 6: return pick_fwd_v<6, kFwdSolo>(fp32w, res);
      default: return pick_fwd_v<4, kFwdSolo>(fp32w, res);
    }
  }
  switch (s.vpt) {
    case 1: return pick_fwd_v<1, kFwdPair>(fp32w, res);
    case 2: return pick_fwd_v<2, kFwdPair>(fp32w, res);
    case 3: return pick_fwd_v<3, kFwdPair>(fp32w, res);
    default: return pick_fwd_v<4, kFwdPair>(fp32w, res);
  }
}


int fwd_blocks_per_sm(const Shape& s, bool fp32w) {
  return blocks_per_sm(pick_fwd(s, fp32w, s.tensors == 2), s.threads, s.smem);
}

cudaError_t launch_fwd(const FwdArgs& a, const Shape& s, bool fp32w, cudaStream_t st) {
  const void* fn = pick_fwd(s, fp32w, a.res != nullptr);
  cudaError_t e = prepare_kernel(fn, s.smem);
  if (e != cudaSuccess) return e;
  FwdArgs copy = a;
  void* args[] = {&copy};
  return launch_pdl(fn, dim3(static_cast<unsigned>(a.P)), dim3(static_cast<unsigned>(s.threads)),
                    s.smem, st, args);
}

}  // namespace rmsn
