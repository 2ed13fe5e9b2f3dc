// rmsn_api.cu -- the C ABI (include/rmsnorm_train.h): argument checks, launch planning,
// and kernel launches.  Never allocates, frees or synchronizes (except the diagnostic
// rmsnorm_train_device_error); every launch goes on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "rmsnorm_train.h"  // include/ (on the include path)
#include "rmsn_launch.h"

namespace rmsn {

// Device error word (bounded waits that gave up), one per device that loads the library.
__device__ unsigned g_err_word = 0u;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxRows = (int64_t{1} << 31) - (int64_t{1} << 16);
// Shared-memory ring bytes per CTA (target): kernels built for two CTAs an SM take 96 KB
// each; "wide" kernels, one CTA an SM, take twice that.
constexpr size_t kRingTarget = 96 * 1024;
constexpr size_t kRingTargetWide = 192 * 1024;
// the tensor-memory class: three stages of its larger row count within this ring
constexpr size_t kRingTargetTm = 200 * 1024;
constexpr size_t kRingTargetSmall = 64 * 1024;
// Forward rows whose group has at least this many threads run one CTA an SM (kFwdSolo).
constexpr int kFwdSoloMinGroup = 64;
// Largest row group of the backward's multi-group class (a multiple of 32, <= 480 / 2).
constexpr int kMultiMaxGroup = 240;
constexpr int kMaxStages = 12;
// The forward keeps at most three stages in flight a CTA: its consumers outrun HBM, so
// every free stage is an outstanding load, and fewer streams per SM make better use of
// the DRAM (measured, one CTA an SM, H = 1536..6144: 3 stages 1-6 % ahead of 6 at large
// T and in the back-to-back clock at T = 16384, 2 stages 10-20 % behind; two CTAs an SM,
// [T,24,256] of 32 heads: 3 stages 8 % ahead of 6).
constexpr int kFwdMaxStages = 3;
constexpr size_t kMaxSmemBytes = 227 * 1024;  // dynamic shared memory a CTA may take
// Deterministic backward: at most kDetSMs x (the CTAs an SM the kernel is built to keep
// resident) dw partials -- a function of the shape only, so the same on every device
// whatever its SM count.  152 is GB300's SM count: there the partition is one wave.
constexpr int kDetSMs = 152;
// Smallest chunk a backward CTA takes, in stages (measured: CTAs of one stage each cut the
// T=64 latency by a quarter against four; no change at large T).
constexpr int kMinStagesPerCta = 1;

std::mutex g_mu;
std::unordered_map<uint64_t, int> g_occ;       // (device, fn, threads, smem) -> blocks/SM
std::unordered_map<uint64_t, bool> g_prepared; // (device, fn) -> smem attribute set
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

uint64_t key(int dev, const void* fn, uint64_t extra) {
  uint64_t h = reinterpret_cast<uint64_t>(fn);
  h ^= (static_cast<uint64_t>(dev) + 0x9e3779b97f4a7c15ull) + (h << 6) + (h >> 2);
  h ^= extra + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
  return h;
}

size_t shared_bytes(const Shape& s, int H, bool bwd) {
  return smem_layout(s.stages, s.tensors, s.groups, H, s.ntg >= 32 ? s.groups : 0,
                     bwd ? s.groups : 0, bwd && bwd_w_in_smem(s.cls, s.vpt) ? H : 0,
                     bwd ? 2 * s.stages : 0)
      .total;
}

Shape make_shape(int H, int tensors, int vpt, bool bwd, bool allow_multi = true,
                 bool tm = false, int tm_min_stages = 3) {
  Shape s{};
  const int nv = H / 8;
  s.vpt = vpt;
  const int per = (nv + s.vpt - 1) / s.vpt;
  if (per <= 8) {
    s.ntg = 8;  // sub-warp groups: four rows a warp
  } else if (per <= 16) {
    s.ntg = 16;  // two rows a warp
  } else {
    s.ntg = ((per + 31) / 32) * 32;
  }
  if (bwd) {
    if (tm)
      s.cls = kBwdTm;
    else if (allow_multi && vpt >= 2 && s.ntg <= kMultiMaxGroup)
      s.cls = kBwdMulti;
    else if (vpt >= 2 && s.ntg >= 32)
      s.cls = kBwdWide;
    else
      s.cls = kBwdNarrow;
  } else {
    // one-warp rows of up to 4 vectors a thread: two CTAs an SM (measured 2-5 % ahead of
    // one CTA of 16 such rows at H = 768 and 1024); larger row groups and the 6-vector
    // build: one CTA an SM
    s.cls = (vpt == 6 || (vpt >= 2 && s.ntg >= kFwdSoloMinGroup)) ? kFwdSolo : kFwdPair;
  }
  // one-CTA-an-SM classes with several row groups fill 512 (forward) or 480 (backward)
  // consumers, the rest 256
  int budget = kMaxConsumerThreads / 2;
  if (!bwd && s.cls == kFwdSolo) budget = fwd_solo_consumers(vpt);
  if (bwd && s.cls == kBwdMulti) budget = kMultiConsumers;
  if (bwd && s.cls == kBwdTm) budget = kTmConsumers;
  s.groups = s.ntg >= budget ? 1 : budget / s.ntg;
  // whole-warp groups: at most 16 (their reduction slots in shared memory)
  if (s.ntg >= 32 && s.groups > 16) s.groups = 16;
  if (bwd && s.cls == kBwdTm) {
    // whole warps of consumers, and as many groups as leave tm_min_stages stages in the
    // ring
    const int step = s.ntg < 32 ? 32 / s.ntg : 1;
    s.groups -= s.groups % step;
    while (s.groups > step &&
           kRingTargetTm / (static_cast<size_t>(tensors) * s.groups * H * 2) <
               static_cast<size_t>(tm_min_stages))
      s.groups -= step;
  }
  s.tensors = tensors;
  s.threads = s.groups * s.ntg + kProducerThreads;
  const size_t stage_bytes = static_cast<size_t>(tensors) * s.groups * H * 2;
  // kernels built for one CTA an SM take the wide ring; forward CTAs of at most 6 warps
  // take a 64 KB ring so that three share an SM when that still leaves four or more
  // stages; the rest take 96 KB (two CTAs an SM)
  const bool one_cta = bwd ? s.cls != kBwdNarrow : s.cls == kFwdSolo;
  size_t target = one_cta ? (s.cls == kBwdTm && bwd ? kRingTargetTm : kRingTargetWide)
                          : kRingTarget;
  if (!bwd && !one_cta && s.threads <= 192 && kRingTargetSmall / stage_bytes >= 4)
    target = kRingTargetSmall;
  int st = static_cast<int>(target / stage_bytes);
  s.stages = st < 2 ? 2 : (st > kMaxStages ? kMaxStages : st);
  if (!bwd && s.stages > kFwdMaxStages) s.stages = kFwdMaxStages;
  s.smem = shared_bytes(s, H, bwd);
  return s;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return RMSN_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return RMSN_ERR_DEVICE;
  return RMSN_OK;
}

// Checks the device generation and caches its SM count and error-word address.
int device_setup(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev]) return RMSN_OK;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RMSN_ERR_CUDA;
  if (major != 10 || minor != 3) return RMSN_ERR_DEVICE;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess || p == nullptr) return RMSN_ERR_CUDA;
  g_sms[dev] = sms;
  g_err_ptr[dev] = static_cast<unsigned*>(p);
  return RMSN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tag of a non-deterministic backward call: nonzero, and different from the last 2^32 - 2
// calls' (the row counter it marks is cleared by each call's finish).
std::atomic<uint32_t> g_call_tag{0};
uint32_t next_call_tag() {
  uint32_t t;
  do {
    t = g_call_tag.fetch_add(1u, std::memory_order_relaxed) + 1u;
  } while (t == 0u);
  return t;
}

// Checks shared by both directions; view strides apply to the strided input only.
int check_view(int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head, int w_dtype) {
  if (T < 0 || nh < 1) return RMSN_ERR_INVALID_ARG;
  if (w_dtype != RMSN_W_BF16 && w_dtype != RMSN_W_FP32) return RMSN_ERR_INVALID_ARG;
  if (H <= 0 || (H % 8) != 0) return RMSN_ERR_INVALID_ARG;
  if (H > kMaxH) return RMSN_ERR_UNSUPPORTED;
  // row indices, plus a stage's worth of rows past the end, stay inside int32
  if (T > 0 && T * static_cast<int64_t>(nh) > kMaxRows) return RMSN_ERR_UNSUPPORTED;
  if (s_tok < 0 || (s_tok % 8) != 0) return RMSN_ERR_INVALID_ARG;
  if (nh > 1 && (s_head < 0 || (s_head % 8) != 0)) return RMSN_ERR_INVALID_ARG;
  return RMSN_OK;
}

bool is_contig(int32_t nh, int32_t H, int64_t s_tok, int64_t s_head) {
  return s_tok == static_cast<int64_t>(nh) * H && (nh == 1 || s_head == H);
}

// Deterministic backward: the partial count, a function of (R, the shape) only.
int det_partials(int32_t R, const Shape& s) {
  const int64_t per = static_cast<int64_t>(s.groups) * kMinStagesPerCta;
  int64_t want = (R + per - 1) / per;
  if (want < 1) want = 1;
  const int64_t cap = static_cast<int64_t>(kDetSMs) * bwd_design_blocks_per_sm(s.cls);
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

// ---- helpers used by the kernel translation units ------------------------------------

// Launch shapes: a thread owns VPT 16-byte column vectors of every row its group takes;
// each kernel's vector count and row-group layout follow from H (and from the residual
// form or dh), chosen for rows in flight within the kernel build's register budget.
Shape fwd_shape(int H, bool residual) {
  const int nv = H / 8;
  const int tensors = residual ? 2 : 1;
  // narrow rows (H <= 512): 4 vectors a lane in 8- or 16-lane groups, two CTAs an SM
  if (nv <= 64) return make_shape(H, tensors, nv >= 4 ? 4 : 1, false);
  // wider rows: whole-warp row groups.  Rows of 2-4 vectors a thread run 512 consumers
  // (they fit 96 registers); rows of 6 vectors a thread, 480 (16 warps, 128 registers).
  // The 6-vector build is taken when it puts a quarter more rows in flight (measured:
  // H = 1536 as 15 one-warp rows 0.67 -> 0.82 of peak against 8 two-warp rows; H = 3072
  // 7 rows against 5 gains 3 %; H = 4096 5 rows against 4 loses 2 %); otherwise the
  // vector count with the most rows in flight, then the most threads busy.  Every choice
  // keeps three ring stages when it can.
  auto group = [nv](int v) { return ((nv + v - 1) / v + 31) / 32 * 32; };
  auto groups = [&](int v) {
    const int gt = group(v), budget = fwd_solo_consumers(v);
    const int g = gt > budget ? 0 : budget / gt;
    return g > 16 ? 16 : g;
  };
  auto busy = [&](int v) { return groups(v) * ((nv + v - 1) / v); };
  auto better = [&](int u, int v) {  // u beats v (v == 0: nothing yet)
    if (v == 0) return true;
    if ((u == 6) != (v == 6)) {
      const int g6 = groups(u == 6 ? u : v), g4 = groups(u == 6 ? v : u);
      const bool six = 4 * g6 > 5 * g4;
      return u == 6 ? six : !six;
    }
    return groups(u) > groups(v) || (groups(u) == groups(v) && busy(u) > busy(v));
  };
  Shape best{}, any{};
  for (int v : {2, 3, 4, 6}) {
    if (groups(v) == 0) continue;
    const Shape s = make_shape(H, tensors, v, false);
    if (better(v, any.vpt)) any = s;
    if (s.stages >= 3 && better(v, best.vpt)) best = s;
  }
  return best.vpt != 0 ? best : any;
}

Shape bwd_shape(int H, bool with_dh) {
  const int nv = H / 8;
  // rows that 240 threads cover with 2 to 4 vectors each (narrow rows in 8- or 16-lane
  // groups): several row groups in one CTA (kBwdMulti); wider rows: see below; H = 8:
  // one-vector lanes, two CTAs an SM (kBwdNarrow)
  auto group = [nv](int v) {  // threads a row group takes (8, 16 or whole warps)
    const int per = (nv + v - 1) / v;
    return per <= 8 ? 8 : (per <= 16 ? 16 : (per + 31) / 32 * 32);
  };
  auto groups = [&](int v) {  // row groups of a multi-group CTA, 0 if a row does not fit
    const int gt = group(v);
    if (gt > kMultiMaxGroup) return 0;
    return (gt < 32 || kMultiConsumers / gt < 16) ? kMultiConsumers / gt : 16;
  };
  auto busy = [&](int v) { return groups(v) * ((nv + v - 1) / v); };  // threads with data
  const int tensors = with_dh ? 3 : 2;
  if (nv < 2) return make_shape(H, tensors, 1, true);
  if (groups(2) > 0 || groups(3) > 0) {
    // the vector count with the most rows in flight, then the most threads busy with row
    // data (measured: rows in flight decide this kernel's bandwidth -- H = 1536 gains 7 %
    // with 7 two-warp rows over 5 three-warp rows); 4-vector threads (weight in shared
    // memory) only while the ring still holds three stages of them
    auto better = [&](int u, int v) {
      return groups(u) != groups(v) ? groups(u) > groups(v) : busy(u) > busy(v);
    };
    const int v = better(3, 2) ? 3 : 2;
    Shape best = make_shape(H, tensors, v, true);
    if (groups(4) > 0 && better(4, v)) {
      const Shape s4 = make_shape(H, tensors, 4, true);
      if (s4.stages >= 3) best = s4;
    }
    // The tensor-memory class where it keeps more rows in flight (its dw state leaves
    // the registers, so 20 warps fit): the vector count with the most rows a stage at
    // three stages (the fewest vectors among equals), then as many rows as keep the
    // multi class's ring depth -- the non-deterministic pool's counter round trips want
    // the deeper ring, and both modes run one program on one shape (measured at H = 1536:
    // 8 rows in 4 stages 4 % ahead of 9 in 3, and of 7 in 4 in the multi class).
    int tv = 0, tg = best.groups;
    for (int u = 2; u <= 4; ++u) {
      if (group(u) > kMultiMaxGroup) continue;
      const Shape t = make_shape(H, tensors, u, true, true, /*tm=*/true);
      if (t.stages >= 3 && t.smem <= kMaxSmemBytes && t.groups > tg) {
        tv = u;
        tg = t.groups;
      }
    }
    if (tv == 0) return best;
    const int depth = best.stages > 3 ? best.stages : 3;
    const Shape t = make_shape(H, tensors, tv, true, true, true, depth);
    return (t.stages >= depth && t.smem <= kMaxSmemBytes && t.groups > best.groups) ? t : best;
  }
  // past 3 x 240 vectors: 4-vector threads in two row groups of up to 240 (H up to 7680)
  // while the ring still holds three stages of them (measured: with two stages the ring
  // runs dry, and one wide group does better), else one wide group
  Shape best = make_shape(H, tensors, nv <= 768 ? 2 : 4, true, /*allow_multi=*/false);
  if (busy(4) > 0) {
    const Shape s = make_shape(H, tensors, 4, true);
    if (s.stages >= 3) best = s;
  }
  // the tensor-memory class with 4-vector rows of up to 304 threads (two or more rows a
  // stage in its 608 consumers) where it keeps more rows in flight at three stages
  const Shape t = make_shape(H, tensors, 4, true, true, /*tm=*/true);
  if (t.ntg <= kTmConsumers / 2 && t.stages >= 3 && t.smem <= kMaxSmemBytes &&
      t.groups > best.groups)
    return t;
  return best;
}

cudaError_t prepare_kernel(const void* fn, size_t smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t k = key(dev, fn, 0);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_prepared.count(k)) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kMaxSmemBytes));
  if (e != cudaSuccess) return e;
  (void)smem;
  std::lock_guard<std::mutex> lk(g_mu);
  g_prepared[k] = true;
  return cudaSuccess;
}

int blocks_per_sm(const void* fn, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const uint64_t k = key(dev, fn, (static_cast<uint64_t>(threads) << 32) ^ smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occ.find(k);
    if (it != g_occ.end()) return it->second;
  }
  if (prepare_kernel(fn, smem) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1)
    n = 1;
  std::lock_guard<std::mutex> lk(g_mu);
  g_occ[k] = n;
  return n;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       void** args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Both backward entry points: rstd given (rstd_out unused), or rstd == nullptr and the
// row pass recomputes it with eps, writing it to rstd_out (the small path computes it into
// rstd_out first and reads it back).
int bwd_common(const void* x, const void* dy, const void* dh, const float* rstd, float eps,
               float* rstd_out, const void* w, int w_dtype, void* dx, float* dw, void* workspace,
               size_t workspace_bytes, int64_t T, int32_t nh, int32_t H, int64_t s_tok,
               int64_t s_head, int deterministic, void* stream) {
  int st = check_view(T, nh, H, s_tok, s_head, w_dtype);
  if (st != RMSN_OK) return st;
  if (!x || !dy || !w || !dx || !dw) return RMSN_ERR_INVALID_ARG;
  if (deterministic != 0 && deterministic != 1) return RMSN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dh) || !aligned16(w) || !aligned16(dx) ||
      !aligned16(dw) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(rstd) & 3u))
    return RMSN_ERR_INVALID_ARG;
  const int64_t R = T * static_cast<int64_t>(nh);

  int dev = 0;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;
  const cudaStream_t stream_ = static_cast<cudaStream_t>(stream);

  const bool fp32w = (w_dtype == RMSN_W_FP32);
  if (bwd_is_small(R)) {  // one launch, no workspace
    BwdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dy = static_cast<const __nv_bfloat16*>(dy);
    a.dh = static_cast<const __nv_bfloat16*>(dh);
    a.rstd = rstd;
    a.eps = eps;
    a.w = w;
    a.dx = static_cast<__nv_bfloat16*>(dx);
    a.map = RowMapArgs{nh, H, s_tok, nh > 1 ? s_head : 0};
    a.R = static_cast<int32_t>(R);
    a.err = g_err_ptr[dev];
    if (rstd == nullptr && R > 0) {  // rstd first, then the one-launch backward reads it
      if (launch_rstd_rows(a, rstd_out, stream_) != cudaSuccess) return RMSN_ERR_CUDA;
      a.rstd = rstd_out;
    }
    return launch_bwd_small(a, dw, fp32w, stream_) == cudaSuccess ? RMSN_OK : RMSN_ERR_CUDA;
  }
  const Shape s = bwd_shape(H, dh != nullptr);
  // deterministic: the partials start at the workspace; non-deterministic: after the row
  // counter
  const size_t ctl_bytes = deterministic ? 0 : kNdCtlBytes;
  float* part = workspace ? reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                                     ctl_bytes)
                          : nullptr;
  int P = 0;
  if (R > 0) {
    // at most 152 x (CTAs an SM of the class) partials in either mode (the deterministic
    // partition; the non-deterministic one is also bounded by this GPU's resident CTAs)
    P = det_partials(static_cast<int32_t>(R), s);
    if (!deterministic) {
      const int occ = bwd_blocks_per_sm(s, fp32w, rstd == nullptr);
      const int64_t cap = static_cast<int64_t>(g_sms[dev]) * (occ > 0 ? occ : 1);
      if (P > cap) P = static_cast<int>(cap);
    }
    const size_t need = ctl_bytes + static_cast<size_t>(P) * 2 * H * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need) return RMSN_ERR_WORKSPACE;

    BwdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dy = static_cast<const __nv_bfloat16*>(dy);
    a.dh = static_cast<const __nv_bfloat16*>(dh);
    a.rstd = rstd;
    a.eps = eps;
    a.rstd_out = rstd_out;
    a.w = w;
    a.dx = static_cast<__nv_bfloat16*>(dx);
    a.part = part;
    a.ctl = deterministic ? nullptr : static_cast<unsigned*>(workspace);
    a.tag = next_call_tag();
    a.map = RowMapArgs{nh, H, s_tok, nh > 1 ? s_head : 0};
    a.R = static_cast<int32_t>(R);
    a.contig = is_contig(nh, H, s_tok, s_head) ? 1 : 0;
    a.groups = s.groups;
    a.ntg = s.ntg;
    a.stages = s.stages;
    a.P = P;
    a.err = g_err_ptr[dev];
    if (launch_bwd_rows(a, s, fp32w, stream_) != cudaSuccess) return RMSN_ERR_CUDA;
  }
  unsigned* ctl = (deterministic || R == 0) ? nullptr : static_cast<unsigned*>(workspace);
  if (launch_dw_finish(part, dw, P, H, ctl, g_sms[dev], stream_) != cudaSuccess)
    return RMSN_ERR_CUDA;
  return RMSN_OK;
}

}  // namespace rmsn

using namespace rmsn;

extern "C" {

const char* rmsnorm_train_status_str(int status) {
  switch (status) {
    case RMSN_OK: return "ok";
    case RMSN_ERR_INVALID_ARG: return "invalid argument";
    case RMSN_ERR_UNSUPPORTED: return "unsupported size";
    case RMSN_ERR_WORKSPACE: return "workspace missing or too small";
    case RMSN_ERR_CUDA: return "CUDA runtime error";
    case RMSN_ERR_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case RMSN_ERR_SCRATCH_LIMIT:
      return "shape needs more than the 16 MiB built-in scratch of rmsnorm_train_bwd_noalloc";
    default: return "unknown status";
  }
}

int rmsnorm_train_fwd(const void* x, const void* residual, const void* w, int w_dtype,
                      void* y, void* h_out, float* rstd, int64_t T, int32_t nh, int32_t H,
                      int64_t s_tok, int64_t s_head, float eps, void* stream) {
  int st = check_view(T, nh, H, s_tok, s_head, w_dtype);
  if (st != RMSN_OK) return st;
  if (!x || !w || !y || !rstd) return RMSN_ERR_INVALID_ARG;
  if ((residual == nullptr) != (h_out == nullptr)) return RMSN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(residual) ||
      !aligned16(h_out) || (reinterpret_cast<uintptr_t>(rstd) & 3u))
    return RMSN_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return RMSN_ERR_INVALID_ARG;
  const int64_t R = T * static_cast<int64_t>(nh);
  if (R == 0) return RMSN_OK;

  int dev = 0;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;

  const bool fp32w = (w_dtype == RMSN_W_FP32);
  const Shape s = fwd_shape(H, residual != nullptr);
  const int occ = fwd_blocks_per_sm(s, fp32w);
  int64_t P = (R + s.groups - 1) / s.groups;
  const int64_t cap = static_cast<int64_t>(g_sms[dev]) * occ;
  if (P > cap) P = cap;

  FwdArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.res = static_cast<const __nv_bfloat16*>(residual);
  a.w = w;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.h = static_cast<__nv_bfloat16*>(h_out);
  a.rstd = rstd;
  a.map = RowMapArgs{nh, H, s_tok, nh > 1 ? s_head : 0};
  a.R = static_cast<int32_t>(R);
  a.contig = is_contig(nh, H, s_tok, s_head) ? 1 : 0;
  a.eps = eps;
  a.groups = s.groups;
  a.ntg = s.ntg;
  a.stages = s.stages;
  a.P = static_cast<int32_t>(P);
  a.err = g_err_ptr[dev];
  return launch_fwd(a, s, fp32w, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RMSN_OK
             : RMSN_ERR_CUDA;
}

size_t rmsnorm_train_bwd_workspace_bytes(int64_t T, int32_t nh, int32_t H, int deterministic) {
  if (check_view(T, nh, H, static_cast<int64_t>(nh) * (H > 0 ? H : 0), H, RMSN_W_BF16) !=
      RMSN_OK)
    return 0;
  const int64_t R = T * static_cast<int64_t>(nh);
  if (R == 0 || bwd_is_small(R)) return 0;  // small inputs take the one-launch path
  // P partials (the launch shape, so the partial count, may differ with and without dh:
  // one size serves both), after the row counter in the non-deterministic mode
  int P = det_partials(static_cast<int32_t>(R), bwd_shape(H, false));
  const int Pd = det_partials(static_cast<int32_t>(R), bwd_shape(H, true));
  if (Pd > P) P = Pd;
  return (deterministic ? 0 : kNdCtlBytes) + static_cast<size_t>(P) * 2 * H * sizeof(float);
}

int rmsnorm_train_bwd(const void* x, const void* dy, const void* dh, const float* rstd,
                      const void* w, int w_dtype, void* dx, float* dw, void* workspace,
                      size_t workspace_bytes, int64_t T, int32_t nh, int32_t H, int64_t s_tok,
                      int64_t s_head, int deterministic, void* stream) {
  if (!rstd) return RMSN_ERR_INVALID_ARG;
  return bwd_common(x, dy, dh, rstd, 0.f, nullptr, w, w_dtype, dx, dw, workspace,
                    workspace_bytes, T, nh, H, s_tok, s_head, deterministic, stream);
}

int rmsnorm_train_bwd_recompute(const void* x, const void* dy, const void* dh, const void* w,
                                int w_dtype, void* dx, float* dw, float* rstd_out,
                                void* workspace, size_t workspace_bytes, int64_t T, int32_t nh,
                                int32_t H, int64_t s_tok, int64_t s_head, float eps,
                                int deterministic, void* stream) {
  if (!rstd_out || (reinterpret_cast<uintptr_t>(rstd_out) & 3u)) return RMSN_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return RMSN_ERR_INVALID_ARG;
  return bwd_common(x, dy, dh, nullptr, eps, rstd_out, w, w_dtype, dx, dw, workspace,
                    workspace_bytes, T, nh, H, s_tok, s_head, deterministic, stream);
}

int rmsnorm_train_launch_plan(int32_t H, int op, int64_t* out, int n_out) {
  if (!out || n_out < 0 || op < RMSN_PLAN_FWD || op > RMSN_PLAN_BWD_ND_DH)
    return RMSN_ERR_INVALID_ARG;
  if (H <= 0 || (H % 8) != 0) return RMSN_ERR_INVALID_ARG;
  if (H > kMaxH) return RMSN_ERR_UNSUPPORTED;
  const bool bwd = op >= RMSN_PLAN_BWD;
  const Shape s = bwd ? bwd_shape(H, op == RMSN_PLAN_BWD_DH || op == RMSN_PLAN_BWD_ND_DH)
                      : fwd_shape(H, op == RMSN_PLAN_FWD_RESIDUAL);
  const int64_t v[RMSN_PLAN_FIELDS] = {
      s.vpt, s.ntg, s.groups, s.stages, s.threads, static_cast<int64_t>(s.smem), s.cls,
      bwd ? bwd_max_threads(s.cls, s.vpt) : fwd_max_threads(s.cls, s.vpt),
      bwd ? bwd_design_blocks_per_sm(s.cls) : fwd_design_blocks_per_sm(s.cls)};
  for (int i = 0; i < n_out && i < RMSN_PLAN_FIELDS; ++i) out[i] = v[i];
  return RMSN_OK;
}

int rmsnorm_train_device_error(unsigned int* flags, int reset) {
  if (!flags) return RMSN_ERR_INVALID_ARG;
  int dev = 0, st;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return RMSN_ERR_CUDA;
  if (cudaMemcpyFromSymbol(flags, g_err_word, sizeof(unsigned)) != cudaSuccess)
    return RMSN_ERR_CUDA;
  if (reset) {
    const unsigned zero = 0u;
    if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(unsigned)) != cudaSuccess)
      return RMSN_ERR_CUDA;
  }
  return RMSN_OK;
}

}  // extern "C"

// ---- backward without caller-provided workspace ----------------------------------------
//
// Some callers cannot allocate device memory where they call the backward: a plugin's
// enqueue callback inside an inference or training runtime that forbids allocation
// there, or a host program with no device allocator of its own to hand out a workspace.
// For them, rmsnorm_train_bwd_noalloc keeps the dw partials in the static array below,
// which every device that loads this library holds until the process exits.  The array
// needs no initial contents: every call writes each partial it later reads.  All calls
// on a device share it, so two calls that overlap on the GPU (different streams, no
// ordering between them) race on it.

namespace rmsn {

constexpr size_t kNoAllocScratchBytes = size_t{16} << 20;  // 16 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on device `dev` (current).  Host code must not use
// the symbol itself as a pointer: on the host it names a stand-in, not device memory.
int noalloc_scratch(int dev, float** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return RMSN_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return RMSN_OK;
}
}  // namespace

}  // namespace rmsn

extern "C" int rmsnorm_train_bwd_noalloc(const void* x, const void* dy, const void* dh,
                                         const float* rstd, const void* w, int w_dtype,
                                         void* dx, float* dw, int64_t T, int32_t nh,
                                         int32_t H, int64_t s_tok, int64_t s_head,
                                         int deterministic, void* stream) {
  int st = check_view(T, nh, H, s_tok, s_head, w_dtype);
  if (st != RMSN_OK) return st;
  if (deterministic != 0 && deterministic != 1) return RMSN_ERR_INVALID_ARG;
  int dev = 0;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;
  const size_t need = rmsnorm_train_bwd_workspace_bytes(T, nh, H, deterministic);
  if (need > kNoAllocScratchBytes) return RMSN_ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  if ((st = noalloc_scratch(dev, &scratch)) != RMSN_OK) return st;
  return rmsnorm_train_bwd(x, dy, dh, rstd, w, w_dtype, dx, dw, scratch, kNoAllocScratchBytes,
                           T, nh, H, s_tok, s_head, deterministic, stream);
}
