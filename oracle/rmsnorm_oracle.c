/*
 * rmsnorm_oracle.c -- plain, slow FP64 CPU oracle for RMSNorm training.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads, links or calls this
 * file: only the tests, the smoke check and the benchmark's CPU baseline do.  It shares
 * no code, header, table or helper with the CUDA library; the two meet only through the
 * seeded inputs that the tests hand to both.
 *
 * What it computes (flashinfer PR #8827 "fix(cake_rmsnorm): sm_100a and sm_107a
 * dw-accuracy backward routes", description: the op contract, and its Measurement
 * section's workload line: eps 1e-6, y / dx / h_new BF16, rstd / dw FP32):
 *
 *   forward, per normalized row (token t, head h) with elements v_j, j = 0..H-1:
 *     residual form only:  v_j := BF16_RNE(x_in_j + res_j)   (h_new, written out)
 *     ms   = (1/H) * sum_j v_j^2
 *     rstd = 1 / sqrt(ms + eps)
 *     y_j  = v_j * rstd * w_j                  (the caller rounds to BF16 to compare)
 *
 *   backward, with r the rstd the backward is handed:
 *     xhat_j = v_j * r,  g_j = dy_j * w_j,  c = (1/H) * sum_j g_j * xhat_j
 *     dx_j   = r * (g_j - xhat_j * c)  [+ dh_j, the residual form's combined gradient]
 *     dw_j   = sum over every row of dy_j * xhat_j
 *
 * Everything is IEEE double, evaluated in the order written above, sequential sums, no
 * blocking or reordering.  Inputs are converted exactly (BF16 and FP32 are subsets of
 * FP64).  Compile with -ffp-contract=off so that no compiler fuses a*b+c: the results
 * are then the same on x86_64 and aarch64.
 *
 * Row addressing (per-head views, same PR, description: "[T,24,256] (strided) and
 * [T,4,256] (contiguous), with a shared w[256]"): row r = t*nh + h of the INPUT
 * activation starts at element t*s_tok + h*s_head; dy, dh and every output are
 * contiguous [T*nh, H].
 *
 * Pinned by tests/test_oracle_pins.py: closed forms (zero row, constant row, a
 * Pythagorean row), a finite-difference gradient check of dx and dw, the identity
 * sum_j x_j*dx_j = rstd^3*eps*sum_j x_j*g_j, special cases (T = 1, dy = 0), exact BF16
 * rounding against hand-made ties, and per-head vs reshaped-plain equality.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- element access ---------------------------------------------------------------- */

/* kind: 0 = BF16 bit pattern (uint16), 1 = FP32, 2 = FP64 */
enum { ORC_BF16 = 0, ORC_F32 = 1, ORC_F64 = 2 };

double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double ld(const void* p, int kind, int64_t i) {
  if (kind == ORC_BF16) return orc_bf16_to_f64(((const uint16_t*)p)[i]);
  if (kind == ORC_F32) return (double)((const float*)p)[i];
  return ((const double*)p)[i];
}

/* Round a double to the nearest BF16 value, ties to even, in ONE rounding step (no
 * detour through FP32, which would round twice).  BF16 = 1 sign, 8 exponent, 7 stored
 * fraction bits: normal numbers have 8 significant bits, the spacing in the binade
 * [2^e, 2^(e+1)) is 2^(e-7); below 2^-126 the spacing is fixed at 2^-133. */
uint16_t orc_f64_to_bf16_rne(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
  double a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  if (a == 0.0) return sign;
  int e = ilogb(a);
  int qexp = (e < -126) ? -133 : e - 7;
  double q = ldexp(a, -qexp);       /* exact: power-of-two scaling inside FP64's range */
  double n = rint(q);               /* default rounding mode: to nearest, ties to even */
  double r = ldexp(n, qexp);        /* exact: n has at most 9 significant bits */
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* overflow -> inf */
  float f = (float)r;               /* exact: r is a BF16 value, hence an FP32 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void orc_round_bf16(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16_rne(v[i]);
}

static int64_t row_base(int64_t r, int32_t nh, int64_t s_tok, int64_t s_head) {
  int64_t t = r / nh, h = r % nh;
  return t * s_tok + h * s_head;
}

/* Loads row r of the forward's normalized input into v[0..H-1]: x itself, or
 * BF16_RNE(x_in + res) for the residual form (the sum of two BF16 values is exact in
 * FP64, so the single rounding here is the whole story).  h_bits, if given, gets the
 * BF16 bit pattern of the residual sum. */
static void load_row(int64_t r, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
                     const void* x, int x_kind, const void* res, int res_kind,
                     double* v, uint16_t* h_bits) {
  int64_t base = row_base(r, nh, s_tok, s_head);
  for (int32_t j = 0; j < H; ++j) {
    double xv = ld(x, x_kind, base + j);
    if (res) {
      uint16_t hb = orc_f64_to_bf16_rne(xv + ld(res, res_kind, base + j));
      if (h_bits) h_bits[j] = hb;
      v[j] = orc_bf16_to_f64(hb);
    } else {
      v[j] = xv;
    }
  }
}

/* ---- forward ----------------------------------------------------------------------- */

/* rows == NULL selects every row 0..T*nh-1 (nrows is then ignored).  For the k-th
 * selected row: rstd[k], y[k*H + j] (if y), h_bits[k*H + j] (if h_bits and res).
 * v_scratch must hold H doubles. */
void orc_fwd(int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
             const void* x, int x_kind, const void* res, int res_kind,
             const void* w, int w_kind, double eps,
             const int64_t* rows, int64_t nrows,
             double* y, double* rstd, uint16_t* h_bits, double* v_scratch) {
  int64_t n = rows ? nrows : T * (int64_t)nh;
  for (int64_t k = 0; k < n; ++k) {
    int64_t r = rows ? rows[k] : k;
    load_row(r, nh, H, s_tok, s_head, x, x_kind, res, res_kind, v_scratch,
             h_bits ? h_bits + k * H : NULL);
    double ss = 0.0;
    for (int32_t j = 0; j < H; ++j) ss += v_scratch[j] * v_scratch[j];
    double ms = ss / (double)H;
    double rs = 1.0 / sqrt(ms + eps);
    rstd[k] = rs;
    if (y)
      for (int32_t j = 0; j < H; ++j) y[k * H + j] = v_scratch[j] * rs * ld(w, w_kind, j);
  }
}

/* ---- backward ---------------------------------------------------------------------- */

/* dx for the selected rows.  x is the forward's normalized input (x, or h for the
 * residual form) under the view strides; dy and dh (nullable) are contiguous [T*nh, H];
 * r_all[row] is the rstd handed to the backward, indexed by global row.  dx[k*H + j].
 * scratch must hold 2*H doubles. */
void orc_bwd_dx(int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
                const void* x, int x_kind, const void* dy, int dy_kind,
                const void* dh, int dh_kind, const double* r_all,
                const void* w, int w_kind,
                const int64_t* rows, int64_t nrows, double* dx, double* scratch) {
  int64_t n = rows ? nrows : T * (int64_t)nh;
  double* xhat = scratch;
  double* g = scratch + H;
  for (int64_t k = 0; k < n; ++k) {
    int64_t r = rows ? rows[k] : k;
    int64_t base = row_base(r, nh, s_tok, s_head);
    double rr = r_all[r];
    for (int32_t j = 0; j < H; ++j) {
      xhat[j] = ld(x, x_kind, base + j) * rr;
      g[j] = ld(dy, dy_kind, r * H + j) * ld(w, w_kind, j);
    }
    double dot = 0.0;
    for (int32_t j = 0; j < H; ++j) dot += g[j] * xhat[j];
    double c = dot / (double)H;
    for (int32_t j = 0; j < H; ++j) {
      double d = rr * (g[j] - xhat[j] * c);
      if (dh) d += ld(dh, dh_kind, r * H + j);
      dx[k * H + j] = d;
    }
  }
}

/* dw[j] = sum over ALL rows r = 0..T*nh-1, in row order, of dy[r][j] * (x[r][j] * r_all[r]). */
void orc_bwd_dw(int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
                const void* x, int x_kind, const void* dy, int dy_kind,
                const double* r_all, double* dw) {
  for (int32_t j = 0; j < H; ++j) dw[j] = 0.0;
  int64_t R = T * (int64_t)nh;
  for (int64_t r = 0; r < R; ++r) {
    int64_t base = row_base(r, nh, s_tok, s_head);
    double rr = r_all[r];
    for (int32_t j = 0; j < H; ++j)
      dw[j] += ld(dy, dy_kind, r * H + j) * (ld(x, x_kind, base + j) * rr);
  }
}
