/*
 * layernorm_oracle.c -- plain, slow FP64 CPU oracle for LayerNorm training (the
 * normalization that sits beside RMSNorm in the ROCm TransformerEngine PR #478
 * microbenchmark tables: "LayerNorm" forward and backward, M rows of hidden_size).
 *
 * TEST INFRASTRUCTURE ONLY, like rmsnorm_oracle.c: nothing on the product path loads it,
 * and it shares no code with any GPU source.  The pages print no formula for LayerNorm;
 * this is the textbook definition, with weight w and bias b:
 *
 *   forward, per row of H elements v_j:
 *     mean = (1/H) * sum_j v_j
 *     var  = (1/H) * sum_j (v_j - mean)^2          (two passes: no E[v^2] - mean^2)
 *     rstd = 1 / sqrt(var + eps)
 *     y_j  = (v_j - mean) * rstd * w_j + b_j       (the caller rounds to BF16 to compare)
 *
 *   backward, with the mean and rstd the backward is handed:
 *     xhat_j = (v_j - mean) * rstd,  g_j = dy_j * w_j
 *     gbar   = (1/H) * sum_j g_j,    c = (1/H) * sum_j g_j * xhat_j
 *     dx_j   = rstd * (g_j - gbar - xhat_j * c)
 *     dw_j   = sum over rows of dy_j * xhat_j,     db_j = sum over rows of dy_j
 *
 * IEEE double, the order written above, sequential sums; rows contiguous [R, H].
 * Compile with -ffp-contract=off (same bits on x86_64 and aarch64).
 *
 * Pinned by tests/test_layernorm_oracle.py: closed forms (constant row, a two-valued row
 * with an exact rstd), finite differences of the loss sum(dy * y) for dx, dw and db, the
 * identities sum_j dx_j = 0 and sum_j dx_j * xhat_j = H * c * eps * rstd^3, special cases
 * (T = 1, dy = 0), and planted-mistake mutants.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { LN_BF16 = 0, LN_F32 = 1, LN_F64 = 2 };

static double ln_ld(const void* p, int kind, int64_t i) {
  if (kind == LN_BF16) {
    uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  if (kind == LN_F32) return (double)((const float*)p)[i];
  return ((const double*)p)[i];
}

/* Forward of rows [0, R): y [R, H] (FP64), mean [R], rstd [R]. */
void ln_fwd(int64_t R, int32_t H, const void* x, int x_kind, const void* w, int w_kind,
            const void* b, int b_kind, double eps, double* y, double* mean, double* rstd) {
  for (int64_t r = 0; r < R; ++r) {
    double s = 0.0;
    for (int32_t j = 0; j < H; ++j) s += ln_ld(x, x_kind, r * H + j);
    const double mu = s / (double)H;
    double ss = 0.0;
    for (int32_t j = 0; j < H; ++j) {
      const double d = ln_ld(x, x_kind, r * H + j) - mu;
      ss += d * d;
    }
    const double var = ss / (double)H;
    const double rs = 1.0 / sqrt(var + eps);
    mean[r] = mu;
    rstd[r] = rs;
    if (y)
      for (int32_t j = 0; j < H; ++j)
        y[r * H + j] = (ln_ld(x, x_kind, r * H + j) - mu) * rs * ln_ld(w, w_kind, j) +
                       ln_ld(b, b_kind, j);
  }
}

/* dx of rows [0, R) (FP64 [R, H]) with the handed mean and rstd; scratch holds 2*H. */
void ln_bwd_dx(int64_t R, int32_t H, const void* x, int x_kind, const void* dy, int dy_kind,
               const double* mean, const double* rstd, const void* w, int w_kind, double* dx,
               double* scratch) {
  double* g = scratch;
  double* xhat = scratch + H;
  for (int64_t r = 0; r < R; ++r) {
    const double mu = mean[r], rs = rstd[r];
    double gs = 0.0, gx = 0.0;
    for (int32_t j = 0; j < H; ++j) {
      g[j] = ln_ld(dy, dy_kind, r * H + j) * ln_ld(w, w_kind, j);
      xhat[j] = (ln_ld(x, x_kind, r * H + j) - mu) * rs;
      gs += g[j];
      gx += g[j] * xhat[j];
    }
    const double gbar = gs / (double)H;
    const double c = gx / (double)H;
    for (int32_t j = 0; j < H; ++j) dx[r * H + j] = rs * (g[j] - gbar - xhat[j] * c);
  }
}

/* dw and db (FP64 [H] each), summed over rows in increasing order. */
void ln_bwd_dw_db(int64_t R, int32_t H, const void* x, int x_kind, const void* dy,
                  int dy_kind, const double* mean, const double* rstd, double* dw,
                  double* db) {
  for (int32_t j = 0; j < H; ++j) {
    dw[j] = 0.0;
    db[j] = 0.0;
  }
  for (int64_t r = 0; r < R; ++r) {
    const double mu = mean[r], rs = rstd[r];
    for (int32_t j = 0; j < H; ++j) {
      const double d = ln_ld(dy, dy_kind, r * H + j);
      dw[j] += d * ((ln_ld(x, x_kind, r * H + j) - mu) * rs);
      db[j] += d;
    }
  }
}
