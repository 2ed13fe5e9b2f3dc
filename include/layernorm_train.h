/*
 * layernorm_train.h -- C ABI of the GB300 (sm_103a) LayerNorm-for-training entry points,
 * built into the same library as rmsnorm_train.h (whose status codes, weight dtypes and
 * conventions -- device pointers, caller-owned buffers, no allocation or synchronization,
 * everything enqueued on `stream` -- apply here too).
 *
 * The operation: LayerNorm with weight w and bias b over rows of H elements, the
 * normalization benchmarked beside RMSNorm in ROCm TransformerEngine PR #478
 * ("Microbenchmarking and CI performance regression test"), normalization tables: forward
 * and backward GB/s for M rows of hidden_size, BF16.  The pages give no formula; this is
 * the textbook definition:
 *
 *   forward   mean = (1/H) sum_j x_j,  var = (1/H) sum_j (x_j - mean)^2     (FP32)
 *             rstd = 1 / sqrt(var + eps)                                    (FP32)
 *             y_j  = BF16(((x_j - mean) * rstd) * w_j + b_j)      round to nearest even
 *   backward  xhat = (x - mean) * rstd,  g = dy * w
 *             dx_j = BF16(rstd * (g_j - mean_k(g_k) - xhat_j * mean_k(g_k * xhat_k)))
 *             dw_j = sum over rows of dy_j * xhat_j,   db_j = sum over rows of dy_j  (FP32)
 *
 * Rows are contiguous: x, y, dy, dx are [R, H]; mean and rstd are [R]; w, b, dw, db [H].
 * When R == 0 the row tensors (x, y, dy, dx, mean, rstd) may be NULL.
 * Alignment: tensor pointers 16-byte aligned except mean and rstd (4-byte; the backward
 * reads them fastest when both are 16-byte aligned); H a multiple of 8.
 * Limits: 0 <= R < 2^31; H a multiple of 8 up to 8192, or a multiple of 16 up to 16384
 * (RMSN_ERR_UNSUPPORTED otherwise).  Above 8192 a cluster of two CTAs takes each row chunk,
 * each CTA owning half of every row's columns.
 * Errors: argument checks return a nonzero status before anything is enqueued;
 * RMSN_ERR_CUDA reports a failed launch.  rmsnorm_train_status_str names a status.
 */
#ifndef LAYERNORM_TRAIN_H
#define LAYERNORM_TRAIN_H

#include <stddef.h>
#include <stdint.h>

#include "rmsnorm_train.h" /* RMSN_OK, RMSN_ERR_*, RMSN_W_BF16, RMSN_W_FP32 */

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Forward: y (BF16), mean and rstd (FP32).
 *   x         BF16 [R, H]
 *   w, b      [H] each, both of dtype wb_dtype (RMSN_W_BF16 or RMSN_W_FP32)
 *   y         BF16 [R, H] out
 *   mean      FP32 [R] out;  rstd  FP32 [R] out
 *   eps       added to the variance inside the square root; finite, >= 0
 * R == 0 returns RMSN_OK with nothing enqueued.
 */
int layernorm_train_fwd(const void* x, const void* w, const void* b, int wb_dtype, void* y,
                        float* mean, float* rstd, int64_t R, int32_t H, float eps,
                        void* stream);

/*
 * Bytes of device workspace layernorm_train_bwd needs: 0 for R == 0.  For
 * deterministic == 0 the size depends on the current device (its SM count); for
 * deterministic != 0 on (R, H) only.  Returns 0 on invalid sizes.
 */
size_t layernorm_train_bwd_workspace_bytes(int64_t R, int32_t H, int deterministic);

/*
 * Backward: dx (BF16), dw and db (FP32): per-CTA partial sums (dw's compensated) added in
 * a fixed order, held to the same per-element budget as the RMSNorm dw (atol 1e-4 +
 * rtol 1e-4 of an FP64 sum).
 *   x          BF16 [R, H], the forward's input
 *   dy         BF16 [R, H], upstream gradient of y
 *   mean, rstd FP32 [R] as returned by the forward
 *   w          [H], dtype wb_dtype (the bias does not enter the backward)
 *   dx         BF16 [R, H] out
 *   dw, db     FP32 [H] out, overwritten (not accumulated); zero-filled when R == 0
 *   workspace  device scratch of >= layernorm_train_bwd_workspace_bytes(...) bytes,
 *              16-byte aligned, no initial contents required, clobbered (may be NULL
 *              when that size is 0)
 *   deterministic  0 or 1: 1 gives bit-identical dw and db run to run and on GPUs of any
 *              SM count; 0 may size the partition to the current GPU.  dx is the same in
 *              both modes, bit for bit.
 */
int layernorm_train_bwd(const void* x, const void* dy, const float* mean, const float* rstd,
                        const void* w, int wb_dtype, void* dx, float* dw, float* db,
                        void* workspace, size_t workspace_bytes, int64_t R, int32_t H,
                        int deterministic, void* stream);

/*
 * The launch plan the library uses for width H (host-only, no CUDA call):
 * op LN_PLAN_FWD or LN_PLAN_BWD; writes min(n_out, LN_PLAN_FIELDS) values to `out` (host
 * memory) in the order: vectors per thread, threads per row group, row groups per CTA,
 * ring stages, threads per CTA, dynamic shared memory bytes, shape class, the class's
 * maximum threads per CTA, CTAs per SM the class is built for, CTAs per row chunk (1, or
 * 2 for a cluster pair; then the other fields describe one CTA of the pair, which owns
 * H/2 columns).
 */
#define LN_PLAN_FWD 0
#define LN_PLAN_BWD 1
#define LN_PLAN_FIELDS 10
int layernorm_train_launch_plan(int32_t H, int op, int64_t* out, int n_out);

/*
 * Device-side error bits of the LayerNorm kernels' bounded waits since the last reset
 * (1: a consumer gave up waiting for staged rows or a row reduction; 2: the producer gave
 * up waiting for a free stage); `flags` is host memory.  Synchronizes the device.
 */
int layernorm_train_device_error(unsigned int* flags, int reset);

#ifdef __cplusplus
}
#endif

#endif /* LAYERNORM_TRAIN_H */
