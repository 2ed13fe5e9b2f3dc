// ln_bwd.cu -- LayerNorm training backward for sm_103a: the dx row pass fused with the dw
// and db partial sums, and the fixed-order finish of both.
//
// Per row, with the forward's mean and rstd r (textbook LayerNorm gradient; the
// normalization benchmarked beside RMSNorm in ROCm TransformerEngine PR #478's tables):
//   d_j = x_j - mean,  xhat_j = d_j * r,  g_j = dy_j * w_j
//   c1  = (1/H) sum_j g_j,   c2 = (1/H) sum_j g_j * xhat_j = (r/H) sum_j g_j * d_j
//   dx_j = BF16(r * (g_j - c1 - xhat_j * c2))
//   dw_j += dy_j * xhat_j,   db_j += dy_j          over every row of every CTA's chunk
//
// The two row sums (sum g, sum g*d) travel together through one reduction per row, so the
// pipeline is the RMSNorm backward's: a producer warp stages x, dy and the rows' mean and
// rstd; phase A of row j forms the partial sums; phase B of row j-1 writes dx and adds the
// row to the thread's dw and db running sums.  dw's running sum carries a Fast2Sum
// compensation term (plain FP32 sums of dy * xhat over a CTA's few hundred rows drift past
// the per-element budget); db's does not need one (its terms are BF16 values, which add
// almost exactly in FP32).  A CTA writes its partial as an unevaluated (hi, lo) FP32 pair
// per column (db: lo = 0); the finish adds the P pairs in a fixed order with TwoSum, so dw
// and db are bit-reproducible for a fixed partition and dx does not depend on the partition
// at all.
#include "ln_common.cuh"
#include "ln_launch.h"

namespace lnorm {

using namespace rmsn;

namespace {

constexpr int kLnFinishCols = 32;
constexpr int kLnFinishSlices = 32;

// Knuth's TwoSum: s + err == a + b exactly, no ordering assumption.
__device__ __forceinline__ float two_sum_ln(float a, float b, float& err) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bp);
  err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
  return s;
}

// Running sum with a Fast2Sum compensation term: acc + cmp tracks the sum of every a*b.
// t = acc + a*b in one fma; acc - t is exact once |acc| >= |a*b| (Fast2Sum), and the
// second fma adds a*b back to it: the addition's error, rounded once, into cmp.
__device__ __forceinline__ void comp_fma_add(f2& acc, f2& cmp, f2 a, f2 b) {
  const f2 t = f2_fma(a, b, acc);
  cmp = f2_add(cmp, f2_fma(a, b, f2_sub(acc, t)));
  acc = t;
}

}  // namespace

// Launch bounds per class (ln_launch.h): kLnBwdMulti up to 480 consumers, kLnBwdTm up to
// 608, kLnBwdWide up to
// 352; each + the producer warp, one CTA an SM.  kPair: the CTA is one of a cluster of two
// that share each row, this one owning the columns [rank*H/2, (rank+1)*H/2) (whole-warp
// row groups only); both CTAs add the row sums of both halves in the same order.
template <int VPT, int kCls, bool kFp32W, bool kPair>
__global__ void __launch_bounds__(ln_max_threads(kCls), 1)
    ln_bwd_rows_kernel(const LnBwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = a.H;
  const int rank = kPair ? static_cast<int>(cluster_cta_rank()) : 0;
  const int Hc = kPair ? (H >> 1) : H;  // the columns this CTA owns
  const int col0 = rank * Hc;
  const int NV = Hc >> 3;
  const int G = a.groups, NTg = a.ntg, S = a.stages;
  const int NW = NTg >> 5;
  const int NWt = kPair ? 2 * NW : NW;  // warps whose partials a row's sums add
  const int SF = kPair ? kLnSlotFloatsPair : kLnSlotFloats;
  const size_t stage_elems = static_cast<size_t>(2) * G * Hc;  // x rows, then dy rows
  const bool red_smem = NTg >= 32;
  // kTm: each consumer thread's dw sums, compensations and db sums live in tensor memory
  // and come to registers one column vector at a time; the weight sits in shared memory
  constexpr bool kTm = kCls == kLnBwdTm;
  const LnSmem L = ln_shape_layout(S, 2, G, H, NTg, kPair, kTm);

  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  uint64_t* redb = reinterpret_cast<uint64_t*>(smem + L.redb);  // [kLnRedBufs][G]
  float* slots = reinterpret_cast<float*>(smem + L.slots);       // [kLnRedBufs][G][SF]
  float* stat = reinterpret_cast<float*>(smem + L.stat);         // [S][2][SP] mean, rstd
  const int SP = ln_stat_stride(G);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

  const int tid = threadIdx.x;
  const int ncons = G * NTg;
  uint32_t* tm_slot = reinterpret_cast<uint32_t*>(smem + L.abort_flag) + 2;
  const uint32_t tm_ncols = kTm ? tmem_alloc_cols(ln_bwd_tm_cols(ncons / 32, VPT)) : 0u;
  const int32_t k = kPair ? static_cast<int32_t>(blockIdx.x >> 1) : blockIdx.x;
  const int32_t r0 = static_cast<int32_t>((static_cast<int64_t>(k) * a.R) / a.P);
  const int32_t r1 = static_cast<int32_t>((static_cast<int64_t>(k + 1) * a.R) / a.P);
  const int32_t nstage = (r1 - r0 + G - 1) / G;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], static_cast<uint32_t>(G * NTg / 32));  // one arrival per warp
    }
    if (red_smem)
      for (int i = 0; i < kLnRedBufs * G; ++i) mbar_init(&redb[i], static_cast<uint32_t>(NWt));
    *abort_flag = 0;
    fence_barrier_init();
  }
  if constexpr (kTm) {
    // consumer warp 0 takes the columns (one CTA an SM); the address reaches the other
    // warps through shared memory
    if (tid < 32) {
      __syncwarp();
      tmem_alloc_warp(tm_slot, tm_ncols);
      tmem_fence_before_sync();
    }
  }
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the peer's barriers exist before any remote use
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  if (tid >= ncons) {  // ---- producer warp ----
    if (tid == ncons) {
      const uint64_t pol = l2_evict_first_policy();
      const bool st_bulk = ((reinterpret_cast<uintptr_t>(a.mean) |
                             reinterpret_cast<uintptr_t>(a.rstd)) & 15u) == 0;
      int32_t j = 0;
      for (; j < nstage; ++j) {
        const int s = j % S;
        if (j >= S &&
            !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((j / S) - 1) & 1u, abort_flag,
                               a.err, kErrProducerWait))
          break;
        const int32_t ra = r0 + j * G;
        const int32_t rb = min(ra + G, r1);
        // The stage's mean and rstd travel with it: the whole 16-byte blocks covering rows
        // [ra, rb) by bulk copies (slot index r - a4), and rows past the arrays' last whole
        // block -- or every row, when either array is not 16-byte aligned -- by 4-byte
        // asynchronous copies that the same barrier tracks (one extra pending arrival,
        // taken before the arrival below).
        const int32_t a4 = ra & ~3;
        const int32_t b4 = st_bulk ? min((rb + 3) & ~3, a.R & ~3) : a4;
        float* md = stat + s * 2 * SP;
        float* rd = md + SP;
        if (rb > b4) {
          for (int32_t r = max(ra, b4); r < rb; ++r) {
            cp_async_4(md + (r - a4), a.mean + r);
            cp_async_4(rd + (r - a4), a.rstd + r);
          }
          cp_async_mbar_arrive(&full[s]);
        }
        const uint32_t st_bytes = static_cast<uint32_t>(b4 - a4) * 4u;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rb - ra) * Hc * 4u + 2u * st_bytes);
        if (st_bytes) {
          bulk_g2s(md, a.mean + a4, st_bytes, &full[s], pol);
          bulk_g2s(rd, a.rstd + a4, st_bytes, &full[s], pol);
        }
        __nv_bfloat16* dst = ring + s * stage_elems;
        if constexpr (kPair) {  // this CTA's half of each row
          copy_half_rows(dst, a.x, H, Hc, col0, ra, rb, &full[s], pol);
          copy_half_rows(dst + static_cast<size_t>(G) * Hc, a.dy, H, Hc, col0, ra, rb, &full[s],
                         pol);
        } else {
          copy_rows_contig(dst, a.x, H, ra, rb, &full[s], pol);
          copy_rows_contig(dst + static_cast<size_t>(G) * H, a.dy, H, ra, rb, &full[s], pol);
        }
      }
      mbar_drain(full, S, j);
    }
    if constexpr (kPair) {
      __syncwarp();
      cluster_sync_all();  // neither CTA exits while its peer may still write its slots
    }
    return;
  }

  // ---- consumers: group g, thread lt owns column vectors c = lt + v*NTg ----
  const int g = tid / NTg;
  const int lt = tid - g * NTg;
  const int wg = lt >> 5, lane = tid & 31;
  Param8<kFp32W> wv[kTm ? 1 : VPT];  // (kTm: the weight is read from shared memory)
  f2 aw[VPT][4], cw[VPT][4], ab[VPT][4];  // dw: sum and compensation; db: sum
  unsigned char* wsm = smem + L.w;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = lt + v * NTg;
    // the weights of the row's column vector col0/8 + c (a pair: this CTA's half)
    if constexpr (!kTm) {
      if (c < NV) load_param8<kFp32W>(a.w, (col0 >> 3) + c, wv[v]);
    }
    if constexpr (!kTm) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        aw[v][q] = f2_splat(0.f);
        cw[v][q] = f2_splat(0.f);
        ab[v][q] = f2_splat(0.f);
      }
    }
  }
  // kTm: vector v's cells at columns tm + 32v: dw sums [0, 8), compensations [8, 16), db
  // sums [16, 24)
  uint32_t tm = 0;
  if constexpr (kTm) {
    // the weight into shared memory as FP32, two planes of float4 (columns 0-3 and 4-7
    // of every vector): conflict-free reads, no conversion per use
    float4* wp = reinterpret_cast<float4*>(wsm);
    for (int c = tid; c < NV; c += ncons) {
      Param8<kFp32W> pw;
      load_param8<kFp32W>(a.w, (col0 >> 3) + c, pw);  // (a pair: this CTA's half)
      const f2 w0 = param_pair<kFp32W>(pw, 0), w1 = param_pair<kFp32W>(pw, 1);
      const f2 w2 = param_pair<kFp32W>(pw, 2), w3 = param_pair<kFp32W>(pw, 3);
      wp[c] = make_float4(f2_lo(w0), f2_hi(w0), f2_lo(w1), f2_hi(w1));
      wp[NV + c] = make_float4(f2_lo(w2), f2_hi(w2), f2_lo(w3), f2_hi(w3));
    }
    named_bar_sync(14, ncons);
    __syncwarp();
    tmem_fence_after_sync();
    const uint32_t w = static_cast<uint32_t>(tid >> 5);
    tm = tmem_warp_addr(*tm_slot, w, (w >> 2) * 32u * VPT);
    float z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      tmem_st16(tm + 32u * v, z);
      tmem_st16(tm + 32u * v + 16u, z);
    }
  }
  // this thread's weight pairs for column vector c (its v-th): FP32 planes in shared
  // memory (kTm) or the registers
  const uint32_t ring32 = smem_u32(smem);
  const uint32_t w32 = ring32 + static_cast<uint32_t>(L.w);
  const uint32_t dy_off = static_cast<uint32_t>(G) * Hc * 2u;  // dy rows after x's in a stage
  auto wvec = [&](int v, int c, f2 (&wq)[4]) {
    if constexpr (kTm) {
      const float4 lo = lds128f_at(w32 + 16u * c);
      const float4 hi = lds128f_at(w32 + 16u * (NV + c));
      wq[0] = f2_make(lo.x, lo.y);
      wq[1] = f2_make(lo.z, lo.w);
      wq[2] = f2_make(hi.x, hi.y);
      wq[3] = f2_make(hi.z, hi.w);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) wq[q] = param_pair<kFp32W>(wv[v], q);
    }
  };
  const float inv_h = 1.0f / static_cast<float>(H);
  const int g0 = red_smem ? g : (tid & ~31) / NTg;
  const int32_t ng = (r1 - r0 > g0) ? (r1 - r0 - g0 + G - 1) / G : 0;

  float sg_carry = 0.f, sgd_carry = 0.f;  // sub-warp groups: row j-1's two sums
  int s_cur = 0, s_prev = 0;  // slot and parity of stage j, slot of stage j-1 (increments,
  uint32_t ph = 0;            // no division by the runtime ring depth)
  for (int32_t j = 0; j <= ng; ++j) {
    float sg_new = 0.f, sgd_new = 0.f;
    // ---- phase A, row j: partials of sum g and sum g*d ----
    if (j < ng) {
      const int32_t row = r0 + j * G + g;
      const int s = s_cur;
      mbar_wait_bounded(&full[s], ph, abort_flag, a.err, kErrConsumerWait);
      f2 ga = f2_splat(0.f), gb = f2_splat(0.f), da = f2_splat(0.f), db2 = f2_splat(0.f);
      if (row < r1) {
        const float nmu = -stat[s * 2 * SP + (row - ((r0 + j * G) & ~3))];
        const uint32_t st = ring32 + 2u * static_cast<uint32_t>(s * stage_elems + g * Hc);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
            const uint4 xv = lds128_at(st + 16u * c);
            const uint4 dv = lds128_at(st + dy_off + 16u * c);
            f2 wq[4];
            wvec(v, c, wq);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const f2 gw = f2_mul(bf2_to_f2(u4_get(dv, q)), wq[q]);
              const f2 dd = bf2_minus(u4_get(xv, q), nmu);
              if (q & 1) {
                gb = f2_add(gb, gw);
                db2 = f2_fma(gw, dd, db2);
              } else {
                ga = f2_add(ga, gw);
                da = f2_fma(gw, dd, da);
              }
            }
          }
        }
      }
      const f2 gs = f2_add(ga, gb), ds = f2_add(da, db2);
      const float pg = f2_lo(gs) + f2_hi(gs);
      const float pgd = f2_lo(ds) + f2_hi(ds);
      if (red_smem) {
        const float wg_s = warp_allsum(pg);
        const float wgd_s = warp_allsum(pgd);
        if (lane == 0) {  // a pair: into both CTAs' slots
          const int rb = (j % kLnRedBufs) * G + g;
          float* slot = slots + rb * SF + 2 * (rank * NW + wg);
          *reinterpret_cast<float2*>(slot) = make_float2(wg_s, wgd_s);
          if constexpr (kPair) {
            const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
            st_peer_f2(peer_addr(slot, peer), wg_s, wgd_s);
            mbar_arrive_peer(peer_addr(&redb[rb], peer));
          }
          mbar_arrive(&redb[rb]);
        }
      } else {
        sg_new = subwarp_allsum(pg, NTg);
        sgd_new = subwarp_allsum(pgd, NTg);
      }
    }
    // ---- phase B, row j-1: dx and the dw, db contributions ----
    if (j >= 1) {
      const int32_t jj = j - 1;
      const int32_t row = r0 + jj * G + g;
      const int s = s_prev;
      float SG = sg_carry, SGD = sgd_carry;
      if (red_smem) {
        const int rb = (jj % kLnRedBufs) * G + g;
        if constexpr (kPair)
          mbar_wait_bounded_cluster(&redb[rb], static_cast<uint32_t>(jj / kLnRedBufs) & 1u,
                                    abort_flag, a.err, kErrConsumerWait);
        else
          mbar_wait_bounded(&redb[rb], static_cast<uint32_t>(jj / kLnRedBufs) & 1u, abort_flag,
                            a.err, kErrConsumerWait);
        const float* sl = slots + rb * SF;
        SG = 0.f;
        SGD = 0.f;
        for (int i = 0; i < NWt; ++i) {  // warp order: the same bits in every thread
          const float2 p = *reinterpret_cast<const float2*>(sl + 2 * i);
          SG += p.x;
          SGD += p.y;
        }
      }
      const bool rv = row < r1;
      // (kTm: every thread of the warp takes part in the tensor-memory traffic, with or
      // without a row)
      if (kTm || rv) {
        const int base = (r0 + jj * G) & ~3;
        const float mu = rv ? stat[s * 2 * SP + (row - base)] : 0.f;
        const float rs = rv ? stat[s * 2 * SP + SP + (row - base)] : 0.f;
        const f2 rs2 = f2_splat(rs);
        const f2 c1 = f2_splat(SG * inv_h);
        // xhat*c2 = d * (r^2 SGD / H): one product of d, so the cancelling terms meet in
        // a single fma
        const f2 ncr2 = f2_splat(-(SGD * (rs * inv_h)) * rs);
        const uint32_t st = ring32 + 2u * static_cast<uint32_t>(s * stage_elems + g * Hc);
        const size_t out_row = static_cast<size_t>(row) * H + col0;
        if constexpr (kTm) {
          __syncwarp();
          tmem_wait_st();  // the previous row's sums are stored before they are loaded
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          const bool live = rv && c < NV;
          float tw[16], tb[8];  // kTm: this vector's dw sums and compensations; db sums
          if constexpr (kTm) {
            tmem_ld16(tm + 32u * v, tw);
            tmem_ld8(tm + 32u * v + 16u, tb);
            tmem_wait_ld();
          }
          if (live) {
            const uint4 xv = lds128_at(st + 16u * c);
            const uint4 dv = lds128_at(st + dy_off + 16u * c);
            f2 wq[4];
            wvec(v, c, wq);
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const f2 d2 = bf2_to_f2(u4_get(dv, q));
              const f2 dd = bf2_minus(u4_get(xv, q), -mu);
              const f2 gw = f2_mul(d2, wq[q]);
              const f2 t = f2_fma(dd, ncr2, f2_sub(gw, c1));  // g - c1 - xhat*c2, over r
              o[q] = f2_to_bf2(f2_mul(t, rs2));
              const f2 ddy = f2_mul(d2, dd);  // dy * xhat = ddy * rstd
              if constexpr (kTm) {
                f2 av = f2_make(tw[2 * q], tw[2 * q + 1]);
                f2 cv = f2_make(tw[8 + 2 * q], tw[9 + 2 * q]);
                comp_fma_add(av, cv, ddy, rs2);
                const f2 bv2 = f2_add(f2_make(tb[2 * q], tb[2 * q + 1]), d2);  // dy
                tw[2 * q] = f2_lo(av);
                tw[2 * q + 1] = f2_hi(av);
                tw[8 + 2 * q] = f2_lo(cv);
                tw[9 + 2 * q] = f2_hi(cv);
                tb[2 * q] = f2_lo(bv2);
                tb[2 * q + 1] = f2_hi(bv2);
              } else {
                comp_fma_add(aw[v][q], cw[v][q], ddy, rs2);
                ab[v][q] = f2_add(ab[v][q], d2);  // dy
              }
            }
            stg128(a.dx + out_row + c * 8, make_uint4(o[0], o[1], o[2], o[3]));
          }
          if constexpr (kTm) {
            __syncwarp();
            tmem_st16(tm + 32u * v, tw);
            tmem_st8(tm + 32u * v + 16u, tb);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
    }
    sg_carry = sg_new;
    sgd_carry = sgd_new;
    s_prev = s_cur;
    if (++s_cur == S) {
      s_cur = 0;
      ph ^= 1u;
    }
  }

  // A column vector's running sums of one quantity (0: dw, with its compensation; 1: db),
  // from the registers or (kTm) from tensor memory: every thread of the warp calls it, so
  // the warp-wide tcgen05 loads stay converged.
  auto sums = [&](int v, int qty, f2 (&acc)[4], f2 (&cmp)[4]) {
    if constexpr (kTm) {
      __syncwarp();
      if (qty == 0) {
        float t[16];
        tmem_ld16(tm + 32u * v, t);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[q] = f2_make(t[2 * q], t[2 * q + 1]);
          cmp[q] = f2_make(t[8 + 2 * q], t[9 + 2 * q]);
        }
      } else {
        float t[8];
        tmem_ld8(tm + 32u * v + 16u, t);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[q] = f2_make(t[2 * q], t[2 * q + 1]);
          cmp[q] = f2_splat(0.f);
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[q] = qty == 0 ? aw[v][q] : ab[v][q];
        cmp[q] = qty == 0 ? cw[v][q] : f2_splat(0.f);
      }
    }
  };
  // kTm: warp 0 frees the columns once every consumer has read its own
  auto release_tmem = [&]() {
    if constexpr (kTm) {
      tmem_fence_before_sync();
      named_bar_sync(13, ncons);
      if (tid < 32) {
        __syncwarp();
        tmem_fence_after_sync();
        tmem_dealloc_warp(*tm_slot, tm_ncols);
      }
    }
  };
  if constexpr (kTm) {
    __syncwarp();
    tmem_wait_st();
  }

  // ---- this CTA's partials: per column (hi, lo) with hi + lo == acc + cmp exactly ----
  // part row 0 (hi) and row 1 (lo), each over dw's H columns then db's H columns
  float* part = a.part + static_cast<size_t>(k) * 4 * H + col0;  // this CTA's columns
  if (G == 1) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = lt + v * NTg;
#pragma unroll
      for (int qty = 0; qty < 2; ++qty) {
        f2 acc[4], cmp[4];
        sums(v, qty, acc, cmp);
        if (c < NV) {
          f2 hi[4], lo[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            hi[q] = f2_add(acc[q], cmp[q]);
            lo[q] = f2_sub(cmp[q], f2_sub(hi[q], acc[q]));
          }
          ulonglong2* ph = reinterpret_cast<ulonglong2*>(part + qty * H + c * 8);
          ulonglong2* pl = reinterpret_cast<ulonglong2*>(part + 2 * H + qty * H + c * 8);
          ph[0] = make_ulonglong2(hi[0].v, hi[1].v);
          ph[1] = make_ulonglong2(hi[2].v, hi[3].v);
          pl[0] = make_ulonglong2(lo[0].v, lo[1].v);
          pl[1] = make_ulonglong2(lo[2].v, lo[3].v);
        }
      }
    }
    release_tmem();
    if constexpr (kPair) {
      __syncwarp();
      cluster_sync_all();
    }
    return;
  }
  // several row groups: combine them through shared memory in group order, dw then db.
  // The ring is free once every consumer is past its loop: each stage was waited on (full)
  // by every group that had a row in it, group 0 included, before that group finished.
  named_bar_sync(15, ncons);
  // cbuf: [G][2][H] (hi, lo), each H-slab as two planes of float4 (columns 0-3 and 4-7 of
  // every vector) so that a warp's stores of one plane are contiguous
  float* cbuf = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int qty = 0; qty < 2; ++qty) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = lt + v * NTg;
      f2 acc[4], cmp[4];
      sums(v, qty, acc, cmp);
      if (c < NV) {
        f2 hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hi[q] = f2_add(acc[q], cmp[q]);
          lo[q] = f2_sub(cmp[q], f2_sub(hi[q], acc[q]));
        }
        ulonglong2* ph = reinterpret_cast<ulonglong2*>(cbuf + (2 * g) * Hc);
        ulonglong2* pl = reinterpret_cast<ulonglong2*>(cbuf + (2 * g + 1) * Hc);
        ph[c] = make_ulonglong2(hi[0].v, hi[1].v);
        ph[NV + c] = make_ulonglong2(hi[2].v, hi[3].v);
        pl[c] = make_ulonglong2(lo[0].v, lo[1].v);
        pl[NV + c] = make_ulonglong2(lo[2].v, lo[3].v);
      }
    }
    named_bar_sync(15, ncons);
    for (int col = tid; col < Hc; col += ncons) {
      const int at = ((col & 7) >> 2) * (4 * NV) + (col >> 3) * 4 + (col & 3);
      float sacc = 0.f, e = 0.f;
      for (int gi = 0; gi < G; ++gi) {
        float err;
        sacc = two_sum_ln(sacc, cbuf[(2 * gi) * Hc + at], err);
        e = __fadd_rn(e, __fadd_rn(err, cbuf[(2 * gi + 1) * Hc + at]));
      }
      const float hi = __fadd_rn(sacc, e);
      part[qty * H + col] = hi;
      part[2 * H + qty * H + col] = __fsub_rn(e, __fsub_rn(hi, sacc));
    }
    named_bar_sync(15, ncons);  // cbuf is rewritten by the next quantity
  }
  release_tmem();
  if constexpr (kPair) {
    __syncwarp();
    cluster_sync_all();
  }
}

// dw[col] (col < H) and db[col - H] (col >= H) = sum over k = 0..P-1 of (hi_k + lo_k), in a
// fixed order: slice i of the kLnFinishSlices slices takes k in [i*P/slices,
// (i+1)*P/slices) in increasing k, then the slice sums combine by a pairwise tree in slice
// order (i with i + stride, stride halving), TwoSum carrying the error terms throughout.
__global__ void __launch_bounds__(kLnFinishCols* kLnFinishSlices)
    ln_finish_kernel(const float* __restrict__ part, float* __restrict__ dw,
                     float* __restrict__ db, int P, int H) {
  __shared__ float sh[kLnFinishSlices][kLnFinishCols];
  __shared__ float se[kLnFinishSlices][kLnFinishCols];
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int cl = threadIdx.x % kLnFinishCols;
  const int sl = threadIdx.x / kLnFinishCols;
  const int col = blockIdx.x * kLnFinishCols + cl;
  const int H2 = 2 * H;
  const int row4 = 4 * H;  // floats of one CTA's partial (P * row4 < 2^31 at every size)
  float s = 0.f, e = 0.f;
  if (col < H2) {
    const int ka = (sl * P) / kLnFinishSlices;
    const int kb = ((sl + 1) * P) / kLnFinishSlices;
    int off = ka * row4 + col;
    int kk = ka;
    for (; kk + 4 <= kb; kk += 4, off += 4 * row4) {
      float hi[4], lo[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        hi[u] = part[off + u * row4];
        lo[u] = part[off + u * row4 + H2];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float err;
        s = two_sum_ln(s, hi[u], err);
        e = __fadd_rn(e, __fadd_rn(err, lo[u]));
      }
    }
    for (; kk < kb; ++kk, off += row4) {
      float err;
      s = two_sum_ln(s, part[off], err);
      e = __fadd_rn(e, __fadd_rn(err, part[off + H2]));
    }
  }
  sh[sl][cl] = s;
  se[sl][cl] = e;
  __syncthreads();
#pragma unroll
  for (int stride = kLnFinishSlices / 2; stride > 0; stride >>= 1) {
    if (sl < stride) {
      float err;
      const float S = two_sum_ln(sh[sl][cl], sh[sl + stride][cl], err);
      se[sl][cl] = __fadd_rn(__fadd_rn(se[sl][cl], se[sl + stride][cl]), err);
      sh[sl][cl] = S;
    }
    __syncthreads();
  }
  if (sl == 0 && col < H2) {
    const float out = __fadd_rn(sh[0][cl], se[0][cl]);
    if (col < H)
      dw[col] = out;
    else
      db[col - H] = out;
  }
}

namespace {

template <int VPT, int kCls, bool kPair>
const void* ln_bwd_ptr_v(bool fp32w) {
  return fp32w ? reinterpret_cast<const void*>(&ln_bwd_rows_kernel<VPT, kCls, true, kPair>)
               : reinterpret_cast<const void*>(&ln_bwd_rows_kernel<VPT, kCls, false, kPair>);
}

// kLnBwdMulti is built for 1 and 2 vectors a thread, kLnBwdWide for 3, kLnBwdTm for 2, 3
// and 4; the pair builds
// (half-rows of 4100..8192 columns) for 2 (multi) and 3 (wide).
const void* pick_ln_bwd(const LnShape& s, bool fp32w) {
  if (s.pair)
    return s.cls == kLnBwdWide ? ln_bwd_ptr_v<3, kLnBwdWide, true>(fp32w)
                               : (s.cls == kLnBwdTm ? ln_bwd_ptr_v<4, kLnBwdTm, true>(fp32w)
                                                    : ln_bwd_ptr_v<2, kLnBwdMulti, true>(fp32w));
  if (s.cls == kLnBwdWide) return ln_bwd_ptr_v<3, kLnBwdWide, false>(fp32w);
  if (s.cls == kLnBwdTm)
    return s.vpt == 2 ? ln_bwd_ptr_v<2, kLnBwdTm, false>(fp32w)
                      : (s.vpt == 3 ? ln_bwd_ptr_v<3, kLnBwdTm, false>(fp32w)
                                    : ln_bwd_ptr_v<4, kLnBwdTm, false>(fp32w));
  return s.vpt == 1 ? ln_bwd_ptr_v<1, kLnBwdMulti, false>(fp32w)
                    : ln_bwd_ptr_v<2, kLnBwdMulti, false>(fp32w);
}

}  // namespace

}  // namespace lnorm

namespace lnorm {

int ln_bwd_blocks_per_sm(const LnShape& s, bool fp32w) {
  return rmsn::blocks_per_sm(pick_ln_bwd(s, fp32w), s.threads, s.smem);
}

cudaError_t ln_launch_bwd_rows(const LnBwdArgs& a, const LnShape& s, bool fp32w,
                               cudaStream_t st) {
  const void* fn = pick_ln_bwd(s, fp32w);
  cudaError_t e = rmsn::prepare_kernel(fn, s.smem);
  if (e != cudaSuccess) return e;
  LnBwdArgs copy = a;
  void* args[] = {&copy};
  if (s.pair)
    return ln_launch_pair(fn, static_cast<unsigned>(a.P), static_cast<unsigned>(s.threads),
                          s.smem, st, args);
  return rmsn::launch_pdl(fn, dim3(static_cast<unsigned>(a.P)),
                          dim3(static_cast<unsigned>(s.threads)), s.smem, st, args);
}

cudaError_t ln_launch_finish(const float* part, float* dw, float* db, int P, int H,
                             cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&ln_finish_kernel);
  void* args[] = {&part, &dw, &db, &P, &H};
  const unsigned grid = static_cast<unsigned>((2 * H + kLnFinishCols - 1) / kLnFinishCols);
  return rmsn::launch_pdl(fn, dim3(grid), dim3(kLnFinishCols * kLnFinishSlices), 0, st, args);
}

}  // namespace lnorm
