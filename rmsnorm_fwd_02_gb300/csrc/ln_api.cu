// ln_api.cu -- the LayerNorm C ABI (include/layernorm_train.h): argument checks, launch
// planning and kernel launches.  Never allocates, frees or synchronizes (except the
// diagnostic layernorm_train_device_error); every launch goes on the caller's stream.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "layernorm_train.h"  // include/ (on the include path)
#include "ln_launch.h"

namespace lnorm {

// Device error word of the LayerNorm kernels' bounded waits, one per device.
__device__ unsigned g_ln_err_word = 0u;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kLnRingTarget = 192 * 1024;  // one CTA an SM
// At most four stages in flight a CTA (measured: the backward at H = 4096 3 % faster than
// with six, the rest unchanged; three slowed the backward at H = 1024 and 8192).
constexpr int kLnMaxStages = 4;
constexpr int kTmemColumns = 512;  // tensor-memory columns of an SM
// Deterministic backward: at most kLnDetSMs partials (the row kernels run one CTA an SM),
// a function of the shape only.  152 is GB300's SM count: there the partition is one wave.
constexpr int kLnDetSMs = 152;

std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return RMSN_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return RMSN_ERR_DEVICE;
  return RMSN_OK;
}

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
  if (cudaGetSymbolAddress(&p, g_ln_err_word) != cudaSuccess || p == nullptr)
    return RMSN_ERR_CUDA;
  g_sms[dev] = sms;
  g_err_ptr[dev] = static_cast<unsigned*>(p);
  return RMSN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Widths: multiples of 8 up to kLnMaxH (one CTA a row chunk), and multiples of 16 up to
// kLnMaxHPair (a CTA pair, each owning a 16-byte-aligned half of every row).
int check_width(int32_t H) {
  if (H <= 0 || (H % 8) != 0) return RMSN_ERR_INVALID_ARG;
  if (H > kLnMaxHPair || (H > kLnMaxH && (H % 16) != 0)) return RMSN_ERR_UNSUPPORTED;
  return RMSN_OK;
}

int check_sizes(int64_t R, int32_t H, int wb_dtype) {
  if (R < 0) return RMSN_ERR_INVALID_ARG;
  if (wb_dtype != RMSN_W_BF16 && wb_dtype != RMSN_W_FP32) return RMSN_ERR_INVALID_ARG;
  const int st = check_width(H);
  if (st != RMSN_OK) return st;
  if (R > INT32_MAX - 1) return RMSN_ERR_UNSUPPORTED;
  return RMSN_OK;
}

// Threads of a row group for `vpt` vectors a thread: 8 or 16 lanes (several rows a warp)
// or whole warps.
int group_threads(int nv, int vpt) {
  const int per = (nv + vpt - 1) / vpt;
  return per <= 8 ? 8 : (per <= 16 ? 16 : (per + 31) / 32 * 32);
}

// The shape of class `cls` with `vpt` vectors a thread for rows of H columns (a pair: each
// CTA owns H/2 of them); groups == 0 if a row does not fit.
LnShape make_shape(int H, int tensors, int vpt, int cls, bool pair) {
  LnShape s{};
  const int Hc = pair ? H / 2 : H;
  const int nv = Hc / 8;
  s.vpt = vpt;
  s.cls = cls;
  s.tensors = tensors;
  s.pair = pair ? 1 : 0;
  s.ntg = group_threads(nv, vpt);
  const int budget = ln_consumers(cls);
  if (s.ntg > budget) return s;
  if (pair && s.ntg < 32) return s;  // a pair exchanges whole warps' partials
  s.groups = budget / s.ntg;  // sub-warp groups: a whole number of warps (budget % 32 == 0)
  if (s.ntg >= 32 && s.groups > kLnMaxWarpsPerGroup) s.groups = kLnMaxWarpsPerGroup;
  if (cls == kLnBwdTm) {
    // the CTA's cells fit the SM's 512 tensor-memory columns (whole warps of consumers)
    const int step = s.ntg < 32 ? 32 / s.ntg : 1;
    while (s.groups > step && ln_bwd_tm_cols(s.groups * s.ntg / 32, vpt) > kTmemColumns)
      s.groups -= step;
    if (ln_bwd_tm_cols(s.groups * s.ntg / 32, vpt) > kTmemColumns) s.groups = 0;
    if (s.groups == 0) return s;
  }
  s.threads = s.groups * s.ntg + kLnProducerThreads;
  const size_t stage_bytes = static_cast<size_t>(tensors) * s.groups * Hc * 2;
  const int st = static_cast<int>(kLnRingTarget / stage_bytes);
  s.stages = st < 2 ? 2 : (st > kLnMaxStages ? kLnMaxStages : st);
  s.smem = ln_shape_layout(s.stages, tensors, s.groups, H, s.ntg, pair, cls == kLnBwdTm).total;
  return s;
}

// Among the candidate builds: the most rows in flight (row groups), then the most threads
// with row data, preferring shapes whose ring still holds three stages.
LnShape pick_shape(int H, int tensors, const int (*cand)[2], int ncand) {
  const bool pair = H > kLnMaxH;
  const int nv = (pair ? H / 2 : H) / 8;
  LnShape best{}, any{};
  auto busy = [nv](const LnShape& s) { return s.groups * ((nv + s.vpt - 1) / s.vpt); };
  auto better = [&](const LnShape& u, const LnShape& v) {
    if (v.groups == 0) return true;
    return u.groups != v.groups ? u.groups > v.groups : busy(u) > busy(v);
  };
  for (int i = 0; i < ncand; ++i) {
    const LnShape s = make_shape(H, tensors, cand[i][0], cand[i][1], pair);
    if (s.groups == 0) continue;
    if (better(s, any)) any = s;
    if (s.stages >= 3 && better(s, best)) best = s;
  }
  return best.groups != 0 ? best : any;
}

// Row chunks of a launch: at most one wave -- of CTAs, or of CTA pairs on two SMs each.
int64_t chunk_cap(int sms, int occ, bool pair) {
  const int64_t ctas = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1);
  return pair ? (ctas / 2 > 0 ? ctas / 2 : 1) : ctas;
}

int bwd_partials(int32_t R, const LnShape& s, bool det, int dev, bool fp32w) {
  int64_t want = (static_cast<int64_t>(R) + s.groups - 1) / s.groups;
  if (want < 1) want = 1;
  int64_t cap;
  if (det) {
    cap = chunk_cap(kLnDetSMs, 1, s.pair != 0);
  } else {
    cap = chunk_cap(g_sms[dev], ln_bwd_blocks_per_sm(s, fp32w), s.pair != 0);
  }
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

LnShape ln_fwd_shape(int H) {
  if (H > kLnMaxH) {
    static const int pair_cand[][2] = {{4, kLnFwdPair}};
    return pick_shape(H, 1, pair_cand, 1);
  }
  static const int cand[][2] = {{1, kLnFwd}, {2, kLnFwd}, {4, kLnFwd}};
  return pick_shape(H, 1, cand, 3);
}

cudaError_t ln_launch_pair(const void* fn, unsigned pairs, unsigned threads, size_t smem,
                           cudaStream_t st, void** args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

LnShape ln_bwd_shape(int H) {
  static const int cand[][2] = {{1, kLnBwdMulti}, {2, kLnBwdMulti}, {3, kLnBwdWide}};
  const LnShape s = pick_shape(H, 2, cand, 3);
  if (H > kLnMaxH) {
    // pair widths: the 4-vector tensor-memory pair build where it keeps more rows in flight
    static const int tp[][2] = {{4, kLnBwdTm}};
    const LnShape t = pick_shape(H, 2, tp, 1);
    return (t.groups > s.groups && t.stages >= 3) ? t : s;
  }
  // the tensor-memory class where it keeps more rows in flight (its column sums leave the
  // registers, so 20 warps fit)
  static const int tmc[][2] = {{2, kLnBwdTm}, {3, kLnBwdTm}, {4, kLnBwdTm}};
  const LnShape t = pick_shape(H, 2, tmc, 3);
  if (t.groups > s.groups && t.stages >= 3) return t;
  return s;
}

}  // namespace lnorm

using namespace lnorm;

extern "C" {

int layernorm_train_fwd(const void* x, const void* w, const void* b, int wb_dtype, void* y,
                        float* mean, float* rstd, int64_t R, int32_t H, float eps,
                        void* stream) {
  int st = check_sizes(R, H, wb_dtype);
  if (st != RMSN_OK) return st;
  // the row tensors may be NULL when there are no rows (nothing is read or written)
  if (!w || !b || (R > 0 && (!x || !y || !mean || !rstd))) return RMSN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(b) || !aligned16(y) || !aligned4(mean) ||
      !aligned4(rstd))
    return RMSN_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return RMSN_ERR_INVALID_ARG;
  if (R == 0) return RMSN_OK;

  int dev = 0;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;

  const bool fp32w = (wb_dtype == RMSN_W_FP32);
  const LnShape s = ln_fwd_shape(H);
  int64_t P = (R + s.groups - 1) / s.groups;  // row chunks (CTAs, or CTA pairs)
  const int64_t cap = chunk_cap(g_sms[dev], ln_fwd_blocks_per_sm(s, fp32w), s.pair != 0);
  if (P > cap) P = cap;

  LnFwdArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.w = w;
  a.b = b;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.mean = mean;
  a.rstd = rstd;
  a.R = static_cast<int32_t>(R);
  a.H = H;
  a.eps = eps;
  a.groups = s.groups;
  a.ntg = s.ntg;
  a.stages = s.stages;
  a.P = static_cast<int32_t>(P);
  a.err = g_err_ptr[dev];
  return ln_launch_fwd(a, s, fp32w, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RMSN_OK
             : RMSN_ERR_CUDA;
}

size_t layernorm_train_bwd_workspace_bytes(int64_t R, int32_t H, int deterministic) {
  if (check_sizes(R, H, RMSN_W_BF16) != RMSN_OK) return 0;
  if (R == 0) return 0;
  const LnShape s = ln_bwd_shape(H);
  int dev = 0;
  int P;
  if (deterministic) {
    P = bwd_partials(static_cast<int32_t>(R), s, true, dev, false);
  } else {
    if (current_device(&dev) != RMSN_OK || device_setup(dev) != RMSN_OK) return 0;
    // the larger of the two weight dtypes' partitions, so one size serves both
    P = bwd_partials(static_cast<int32_t>(R), s, false, dev, false);
    const int P2 = bwd_partials(static_cast<int32_t>(R), s, false, dev, true);
    if (P2 > P) P = P2;
  }
  return static_cast<size_t>(P) * 4 * H * sizeof(float);
}

int layernorm_train_bwd(const void* x, const void* dy, const float* mean, const float* rstd,
                        const void* w, int wb_dtype, void* dx, float* dw, float* db,
                        void* workspace, size_t workspace_bytes, int64_t R, int32_t H,
                        int deterministic, void* stream) {
  int st = check_sizes(R, H, wb_dtype);
  if (st != RMSN_OK) return st;
  // the row tensors may be NULL when there are no rows (dw and db are still zero-filled)
  if (!w || !dw || !db || (R > 0 && (!x || !dy || !mean || !rstd || !dx)))
    return RMSN_ERR_INVALID_ARG;
  if (deterministic != 0 && deterministic != 1) return RMSN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(w) || !aligned16(dx) || !aligned16(dw) ||
      !aligned16(db) || !aligned16(workspace) || !aligned4(mean) || !aligned4(rstd))
    return RMSN_ERR_INVALID_ARG;

  int dev = 0;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;
  const cudaStream_t stream_ = static_cast<cudaStream_t>(stream);

  const bool fp32w = (wb_dtype == RMSN_W_FP32);
  int P = 0;
  if (R > 0) {
    const LnShape s = ln_bwd_shape(H);
    P = bwd_partials(static_cast<int32_t>(R), s, deterministic != 0, dev, fp32w);
    const size_t need = static_cast<size_t>(P) * 4 * H * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need) return RMSN_ERR_WORKSPACE;

    LnBwdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dy = static_cast<const __nv_bfloat16*>(dy);
    a.mean = mean;
    a.rstd = rstd;
    a.w = w;
    a.dx = static_cast<__nv_bfloat16*>(dx);
    a.part = static_cast<float*>(workspace);
    a.R = static_cast<int32_t>(R);
    a.H = H;
    a.groups = s.groups;
    a.ntg = s.ntg;
    a.stages = s.stages;
    a.P = P;
    a.err = g_err_ptr[dev];
    if (ln_launch_bwd_rows(a, s, fp32w, stream_) != cudaSuccess) return RMSN_ERR_CUDA;
  }
  if (ln_launch_finish(static_cast<const float*>(workspace), dw, db, P, H, stream_) !=
      cudaSuccess)
    return RMSN_ERR_CUDA;
  return RMSN_OK;
}

int layernorm_train_launch_plan(int32_t H, int op, int64_t* out, int n_out) {
  if (!out || n_out < 0 || (op != LN_PLAN_FWD && op != LN_PLAN_BWD)) return RMSN_ERR_INVALID_ARG;
  const int st = check_width(H);
  if (st != RMSN_OK) return st;
  const LnShape s = op == LN_PLAN_BWD ? ln_bwd_shape(H) : ln_fwd_shape(H);
  const int64_t v[LN_PLAN_FIELDS] = {s.vpt,  s.ntg, s.groups, s.stages, s.threads,
                                     static_cast<int64_t>(s.smem), s.cls,
                                     ln_max_threads(s.cls), 1, s.pair ? 2 : 1};
  for (int i = 0; i < n_out && i < LN_PLAN_FIELDS; ++i) out[i] = v[i];
  return RMSN_OK;
}

int layernorm_train_device_error(unsigned int* flags, int reset) {
  if (!flags) return RMSN_ERR_INVALID_ARG;
  int dev = 0, st;
  if ((st = current_device(&dev)) != RMSN_OK) return st;
  if ((st = device_setup(dev)) != RMSN_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return RMSN_ERR_CUDA;
  if (cudaMemcpyFromSymbol(flags, g_ln_err_word, sizeof(unsigned)) != cudaSuccess)
    return RMSN_ERR_CUDA;
  if (reset) {
    const unsigned zero = 0u;
    if (cudaMemcpyToSymbol(g_ln_err_word, &zero, sizeof(unsigned)) != cudaSuccess)
      return RMSN_ERR_CUDA;
  }
  return RMSN_OK;
}

}  // extern "C"
