// ln_fwd.cu -- LayerNorm training forward for sm_103a.
//
// Per row of H elements (LayerNorm with weight w and bias b, the normalization benchmarked
// beside RMSNorm in ROCm TransformerEngine PR #478's normalization tables; the pages give
// no formula, so this is the textbook one):
//   mean = (1/H) sum_j x_j,   var = (1/H) sum_j (x_j - mean)^2,   rstd = 1/sqrt(var + eps)
//   y_j  = BF16(((x_j - mean) * rstd) * w_j + b_j)      (FP32, one fma, RNE to BF16)
//
// Both statistics in one reduction per row: each thread forms, for its own elements of the
// row shifted by K (the row's first element), their sum S and the sum M of their squared
// deviations from their own mean (two passes over its registers), and the threads'
// (count n, S, M) triples merge pairwise by Chan, Golub and LeVeque's update (1979):
//   S = S_a + S_b,   M = M_a + M_b + (n_b S_a - n_a S_b)^2 / (n_a n_b (n_a + n_b)).
// Then mean = K + S*(1/H) and var = M*(1/H) (1/H correctly rounded: exact for H a power
// of 2, else one more rounding than a division).  Unlike sum(x^2) - H*mean^2 this keeps
// the variance's accuracy when |mean| >> std; unlike a two-pass variance over the whole
// row it needs one
// reduction, so the row pipeline is the RMSNorm forward's: the producer warp stages rows
// into the ring, and split-phase rows let the reduction of row j overlap phase B
// (normalize and store) of row j-1.
#include "ln_common.cuh"
#include "ln_launch.h"

namespace lnorm {

using namespace rmsn;

namespace {

constexpr unsigned kFullMask = 0xffffffffu;

// The row's first element as FP32: the shift K of the row's statistics.  Taking the sums
// of x - K (exact in FP32 when the BF16 values x and K are within a factor 2^15 of each
// other or one is zero, else rounded once) keeps the merge's
// rounding error proportional to |mean - K| / std instead of |mean| / std: the pairwise
// update is first-order in that ratio (Chan, Golub and LeVeque, 1983), and K is one of the
// row's own values.
__device__ __forceinline__ float row_shift(const __nv_bfloat16* xs) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(xs)) << 16);
}

// The same for a CTA of a pair, from the row's staged 16-byte head (element 0 in the low
// half of the first word).
__device__ __forceinline__ float head_shift(const uint4* h) {
  return __uint_as_float(h->x << 16);
}

// Merges (S, M) over an aligned block of W lanes (W = 8, 16 or 32) by the pairwise update.
// `n` is this lane's element count.  Both partners of a step evaluate the same expression
// from the same two operands (addition and multiplication commute, and a - b is exactly
// -(b - a)), so every lane of the block ends with the same bits.  With `uniform` (every
// lane of the warp has the same count: warp-uniform) each step merges equal counts, and
// the factor n_b^2 / (n_a n_b (n_a + n_b)) is 1/(2n): q0 = 1/(2 n0), halved per step, no
// division.  Otherwise the counts travel with the sums and the factor is divided out.
template <int W>
__device__ __forceinline__ void stat_butterfly_w(float& S, float& M, float n, float q0,
                                                 bool uniform) {
  if (uniform) {
    float q = q0;
#pragma unroll
    for (int o = W >> 1; o > 0; o >>= 1) {
      const float Sb = __shfl_xor_sync(kFullMask, S, o);
      const float Mb = __shfl_xor_sync(kFullMask, M, o);
      const float d = __fsub_rn(S, Sb);
      const float corr = __fmul_rn(__fmul_rn(d, d), q);
      q = __fmul_rn(q, 0.5f);
      S = __fadd_rn(S, Sb);
      M = __fadd_rn(__fadd_rn(M, Mb), corr);
    }
  } else {
#pragma unroll
    for (int o = W >> 1; o > 0; o >>= 1) {
      const float Sb = __shfl_xor_sync(kFullMask, S, o);
      const float Mb = __shfl_xor_sync(kFullMask, M, o);
      const float nb = __shfl_xor_sync(kFullMask, n, o);
      const float nn = __fadd_rn(n, nb);
      const float d = __fsub_rn(__fmul_rn(nb, S), __fmul_rn(n, Sb));
      const float corr = (n > 0.f && nb > 0.f)
                             ? __fdiv_rn(__fmul_rn(d, d), __fmul_rn(__fmul_rn(n, nb), nn))
                             : 0.f;
      n = nn;
      S = __fadd_rn(S, Sb);
      M = __fadd_rn(__fadd_rn(M, Mb), corr);
    }
  }
}

// (the block width as a template argument: the steps unroll)
__device__ __forceinline__ void stat_butterfly(float& S, float& M, float n, float q0,
                                               bool uniform, int W) {
  if (W == 32)
    stat_butterfly_w<32>(S, M, n, q0, uniform);
  else if (W == 16)
    stat_butterfly_w<16>(S, M, n, q0, uniform);
  else
    stat_butterfly_w<8>(S, M, n, q0, uniform);
}

}  // namespace

// One build per vector count and parameter dtype; one CTA an SM, up to 608 consumers +
// the producer warp (20 warps: 96 registers a thread).  kPair (class kLnFwdPair, also up to
// 608 consumers, 4-vector threads): the CTA is one of a cluster of two that share each
// row, this one owning the columns [rank*H/2, (rank+1)*H/2) (whole-warp row groups only);
// the two CTAs merge both halves' warp statistics in the same order, so they compute the
// same mean and rstd.
template <int VPT, bool kFp32W, bool kPair>
__global__ void __launch_bounds__(ln_max_threads(kPair ? kLnFwdPair : kLnFwd), 1)
    ln_fwd_kernel(const LnFwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = a.H;
  const int rank = kPair ? static_cast<int>(cluster_cta_rank()) : 0;
  const int Hc = kPair ? (H >> 1) : H;  // the columns this CTA owns
  const int col0 = rank * Hc;
  const int NV = Hc >> 3;
  const int G = a.groups, NTg = a.ntg, S = a.stages;
  const int NW = NTg >> 5;
  const int NWt = kPair ? 2 * NW : NW;  // warps whose partials a row's statistics merge
  const int SF = kPair ? kLnSlotFloatsPair : kLnSlotFloats;
  const size_t stage_elems = static_cast<size_t>(G) * Hc;
  const bool red_smem = NTg >= 32;  // else sub-warp groups: shuffles only
  const LnSmem L = ln_shape_layout(S, 1, G, H, NTg, kPair);

  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  uint64_t* redb = reinterpret_cast<uint64_t*>(smem + L.redb);  // [kLnRedBufs][G]
  float* slots = reinterpret_cast<float*>(smem + L.slots);       // [kLnRedBufs][G][SF]
  uint4* head = reinterpret_cast<uint4*>(smem + L.head);          // [S][G] (pair)
  float* wtab = reinterpret_cast<float*>(smem + L.wtab);         // [3][kLnWtab]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

  const int tid = threadIdx.x;
  const int ncons = G * NTg;
  const int32_t k = kPair ? static_cast<int32_t>(blockIdx.x >> 1) : blockIdx.x;
  const int32_t r0 = static_cast<int32_t>((static_cast<int64_t>(k) * a.R) / a.P);
  const int32_t r1 = static_cast<int32_t>((static_cast<int64_t>(k + 1) * a.R) / a.P);
  const int32_t nstage = (r1 - r0 + G - 1) / G;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], static_cast<uint32_t>(G * NTg / 32));  // one arrival per warp
    }
    if (red_smem) {
      for (int i = 0; i < kLnRedBufs * G; ++i) mbar_init(&redb[i], static_cast<uint32_t>(NWt));
      // per warp of a group (of both CTAs of a pair, rank 0's first: the two halves have
      // the same layout): its element count c, the count of the warps before it, and the
      // merge factor 1/(pre * c * (pre + c)) (0 for the first warp)
      float pre = 0.f;
      for (int wt = 0; wt < NWt; ++wt) {
        const int w = wt % NW;
        int cnt = 0;
        for (int v = 0; v < VPT; ++v) {
          const int left = NV - v * NTg - 32 * w;
          cnt += left <= 0 ? 0 : (left >= 32 ? 32 : left);
        }
        const float c = 8.f * static_cast<float>(cnt);
        wtab[wt] = c;
        wtab[kLnWtab + wt] = pre;
        wtab[2 * kLnWtab + wt] =
            (pre > 0.f && c > 0.f)
                ? static_cast<float>(1.0 / (static_cast<double>(pre) * c * (pre + c)))
                : 0.f;
        pre += c;
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the peer's barriers exist before any remote use
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  if (tid >= ncons) {  // ---- producer warp ----
    if (tid == ncons) {
      const uint64_t pol = l2_evict_first_policy();
      int32_t j = 0;
      for (; j < nstage; ++j) {
        const int s = j % S;
        if (j >= S &&
            !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((j / S) - 1) & 1u, abort_flag,
                               a.err, kErrProducerWait))
          break;
        const int32_t ra = r0 + j * G;
        const int32_t rb = min(ra + G, r1);
        if constexpr (kPair) {
          // this CTA's half of each row, and each row's first 16 bytes (the shift)
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rb - ra) * (Hc * 2u + 16u));
          copy_half_rows(ring + s * stage_elems, a.x, H, Hc, col0, ra, rb, &full[s], pol);
          for (int32_t r = ra; r < rb; ++r)
            bulk_g2s(&head[s * G + (r - ra)], a.x + static_cast<int64_t>(r) * H, 16u, &full[s],
                     pol);
        } else {
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rb - ra) * H * 2u);
          copy_rows_contig(ring + s * stage_elems, a.x, H, ra, rb, &full[s], pol);
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
  // w and b of this CTA's columns in shared memory as FP32, four planes of float4 (w
  // columns 0-3 and 4-7 of every vector, then b's), read per use: conflict-free, and no
  // registers held across rows
  float4* wb = reinterpret_cast<float4*>(smem + L.w);
  for (int c = tid; c < NV; c += ncons) {
    Param8<kFp32W> pw, pb;
    load_param8<kFp32W>(a.w, (col0 >> 3) + c, pw);
    load_param8<kFp32W>(a.b, (col0 >> 3) + c, pb);
    const f2 w0 = param_pair<kFp32W>(pw, 0), w1 = param_pair<kFp32W>(pw, 1);
    const f2 w2 = param_pair<kFp32W>(pw, 2), w3 = param_pair<kFp32W>(pw, 3);
    const f2 b0 = param_pair<kFp32W>(pb, 0), b1 = param_pair<kFp32W>(pb, 1);
    const f2 b2 = param_pair<kFp32W>(pb, 2), b3 = param_pair<kFp32W>(pb, 3);
    wb[c] = make_float4(f2_lo(w0), f2_hi(w0), f2_lo(w1), f2_hi(w1));
    wb[NV + c] = make_float4(f2_lo(w2), f2_hi(w2), f2_lo(w3), f2_hi(w3));
    wb[2 * NV + c] = make_float4(f2_lo(b0), f2_hi(b0), f2_lo(b1), f2_hi(b1));
    wb[3 * NV + c] = make_float4(f2_lo(b2), f2_hi(b2), f2_lo(b3), f2_hi(b3));
  }
  named_bar_sync(14, ncons);
  int nvec = 0;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = lt + v * NTg;
    if (c < NV) {
      ++nvec;
    }
  }
  const float n_lane = 8.f * static_cast<float>(nvec);
  const float inv_n = nvec ? 1.0f / n_lane : 0.f;  // 1/(2 n_lane) = inv_n / 2 exactly
  const bool uniform = __all_sync(kFullMask, nvec == __shfl_sync(kFullMask, nvec, 0));
  const int W = NTg < 32 ? NTg : 32;
  const float hf = static_cast<float>(H);  // exact for H < 2^24
  const float inv_h = 1.0f / hf;           // correctly rounded; exact for H a power of 2
  // Rows of this warp's first group: every lane of a warp runs the same iterations (the
  // shuffles need them all); groups past the chunk's end skip the row work.
  const int g0 = red_smem ? g : (tid & ~31) / NTg;
  const int32_t ng = (r1 - r0 > g0) ? (r1 - r0 - g0 + G - 1) / G : 0;

  float s_carry = 0.f, m_carry = 0.f;  // sub-warp groups: row j-1's merged statistics
  int s_cur = 0, s_prev = 0;  // slot and parity of stage j, slot of stage j-1 (increments,
  uint32_t ph = 0;            // no division by the runtime ring depth)
  for (int32_t j = 0; j <= ng; ++j) {
    float St = 0.f, Mt = 0.f;
    // ---- phase A, row j: this thread's sum and sum of squared deviations ----
    if (j < ng) {
      const int32_t row = r0 + j * G + g;
      const int s = s_cur;
      mbar_wait_bounded(&full[s], ph, abort_flag, a.err, kErrConsumerWait);
      if (row < r1) {
        const __nv_bfloat16* xs = ring + s * stage_elems + static_cast<size_t>(g) * Hc;
        // statistics of x - K, K the row's first element (one value for the whole group,
        // and for both CTAs of a pair)
        // (x - K: the mixed-precision fma reads the staged BF16 words directly)
        const float nK = -(kPair ? head_shift(&head[s * G + g]) : row_shift(xs));
        uint4 xr[VPT];
        f2 s0 = f2_splat(0.f), s1 = f2_splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          xr[v] = make_uint4(0u, 0u, 0u, 0u);
          if (c < NV) {
            xr[v] = lds128_at(smem_u32(xs) + 16u * c);
            s0 = f2_add(s0, bf2_minus(xr[v].x, nK));
            s1 = f2_add(s1, bf2_minus(xr[v].y, nK));
            s0 = f2_add(s0, bf2_minus(xr[v].z, nK));
            s1 = f2_add(s1, bf2_minus(xr[v].w, nK));
          }
        }
        const f2 sp = f2_add(s0, s1);
        St = f2_lo(sp) + f2_hi(sp);
        const f2 m2 = f2_splat(St * inv_n);
        f2 q0a = f2_splat(0.f), q1a = f2_splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const f2 e = f2_sub(bf2_minus(u4_get(xr[v], q), nK), m2);
              if (q & 1)
                q1a = f2_fma(e, e, q1a);
              else
                q0a = f2_fma(e, e, q0a);
            }
          }
        }
        const f2 qp = f2_add(q0a, q1a);
        Mt = f2_lo(qp) + f2_hi(qp);
      }
    }
    // ---- phase B, row j-1: mean, rstd, y ----
    // The staged vectors go to registers and the stage is released at once; then the
    // row's merged statistics are awaited (normally long complete), and row j's lane merge
    // runs inside B's arithmetic.
    if (j >= 1) {
      const int32_t jj = j - 1;
      const int32_t row = r0 + jj * G + g;
      const int s = s_prev;
      const bool valid = row < r1;
      const __nv_bfloat16* xs = ring + s * stage_elems + static_cast<size_t>(g) * Hc;
      uint4 hv[VPT];
      const float K = !valid ? 0.f : (kPair ? head_shift(&head[s * G + g]) : row_shift(xs));
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = lt + v * NTg;
        hv[v] = make_uint4(0u, 0u, 0u, 0u);
        if (valid && c < NV) hv[v] = lds128_at(smem_u32(xs) + 16u * c);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp has its vectors of the stage
      float Sg = s_carry, Mg = m_carry;
      if (red_smem) {
        const int rb = (jj % kLnRedBufs) * G + g;
        if constexpr (kPair)
          mbar_wait_bounded_cluster(&redb[rb], static_cast<uint32_t>(jj / kLnRedBufs) & 1u,
                                    abort_flag, a.err, kErrConsumerWait);
        else
          mbar_wait_bounded(&redb[rb], static_cast<uint32_t>(jj / kLnRedBufs) & 1u, abort_flag,
                            a.err, kErrConsumerWait);
        // the warps' partials merged in warp order: the same bits in every thread (of both
        // CTAs of a pair)
        const float* sl = slots + rb * SF;
        Sg = sl[0];
        Mg = sl[1];
        for (int i = 1; i < NWt; ++i) {
          const float2 p = *reinterpret_cast<const float2*>(sl + 2 * i);
          const float d = __fsub_rn(__fmul_rn(wtab[i], Sg), __fmul_rn(wtab[kLnWtab + i], p.x));
          const float corr = __fmul_rn(__fmul_rn(d, d), wtab[2 * kLnWtab + i]);
          Sg = __fadd_rn(Sg, p.x);
          Mg = __fadd_rn(__fadd_rn(Mg, p.y), corr);
        }
      }
      if (j < ng) stat_butterfly(St, Mt, n_lane, 0.5f * inv_n, uniform, W);
      if (valid) {
        const float mean = __fadd_rn(K, __fmul_rn(Sg, inv_h));
        const float rs = __frsqrt_rn(__fadd_rn(__fmul_rn(Mg, inv_h), a.eps));
        const float nmean = -mean;
        const f2 rs2 = f2_splat(rs);
        const size_t out_row = static_cast<size_t>(row) * H + col0;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int c = lt + v * NTg;
          if (c < NV) {
            const float4 wa = wb[c], wc = wb[NV + c], ba = wb[2 * NV + c], bc = wb[3 * NV + c];
            const f2 wq[4] = {f2_make(wa.x, wa.y), f2_make(wa.z, wa.w), f2_make(wc.x, wc.y),
                              f2_make(wc.z, wc.w)};
            const f2 bq[4] = {f2_make(ba.x, ba.y), f2_make(ba.z, ba.w), f2_make(bc.x, bc.y),
                              f2_make(bc.z, bc.w)};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const f2 xh = f2_mul(bf2_minus(u4_get(hv[v], q), nmean), rs2);
              o[q] = f2_to_bf2(f2_fma(xh, wq[q], bq[q]));
            }
            stg128(a.y + out_row + c * 8, make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
        if (lt == 0 && rank == 0) {
          a.mean[row] = mean;
          a.rstd[row] = rs;
        }
      }
    } else if (j < ng) {
      stat_butterfly(St, Mt, n_lane, 0.5f * inv_n, uniform, W);
    }
    // ---- publish row j's per-warp statistics (a pair: into both CTAs' slots) ----
    if (j < ng && red_smem && lane == 0) {
      const int rb = (j % kLnRedBufs) * G + g;
      const int wi = rank * NW + wg;
      float* slot = slots + rb * SF + 2 * wi;
      *reinterpret_cast<float2*>(slot) = make_float2(St, Mt);
      if constexpr (kPair) {
        const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
        st_peer_f2(peer_addr(slot, peer), St, Mt);
        mbar_arrive_peer(peer_addr(&redb[rb], peer));
      }
      mbar_arrive(&redb[rb]);
    }
    s_carry = St;
    m_carry = Mt;
    s_prev = s_cur;
    if (++s_cur == S) {
      s_cur = 0;
      ph ^= 1u;
    }
  }
  if constexpr (kPair) {
    __syncwarp();
    cluster_sync_all();  // neither CTA exits while its peer may still write its slots
  }
}

namespace {

template <int VPT, bool kPair>
const void* ln_fwd_ptr_v(bool fp32w) {
  return fp32w ? reinterpret_cast<const void*>(&ln_fwd_kernel<VPT, true, kPair>)
               : reinterpret_cast<const void*>(&ln_fwd_kernel<VPT, false, kPair>);
}

// built for 1, 2 and 4 vectors a thread; the pair build (half-rows of 4104..8192
// columns) for 4
const void* pick_ln_fwd(const LnShape& s, bool fp32w) {
  if (s.pair) return ln_fwd_ptr_v<4, true>(fp32w);
  switch (s.vpt) {
    case 1: return ln_fwd_ptr_v<1, false>(fp32w);
    case 2: return ln_fwd_ptr_v<2, false>(fp32w);
    default: return ln_fwd_ptr_v<4, false>(fp32w);
  }
}

}  // namespace

}  // namespace lnorm

namespace lnorm {

int ln_fwd_blocks_per_sm(const LnShape& s, bool fp32w) {
  return rmsn::blocks_per_sm(pick_ln_fwd(s, fp32w), s.threads, s.smem);
}

cudaError_t ln_launch_fwd(const LnFwdArgs& a, const LnShape& s, bool fp32w, cudaStream_t st) {
  const void* fn = pick_ln_fwd(s, fp32w);
  cudaError_t e = rmsn::prepare_kernel(fn, s.smem);
  if (e != cudaSuccess) return e;
  LnFwdArgs copy = a;
  void* args[] = {&copy};
  if (s.pair)
    return ln_launch_pair(fn, static_cast<unsigned>(a.P), static_cast<unsigned>(s.threads),
                          s.smem, st, args);
  return rmsn::launch_pdl(fn, dim3(static_cast<unsigned>(a.P)),
                          dim3(static_cast<unsigned>(s.threads)), s.smem, st, args);
}

}  // namespace lnorm
