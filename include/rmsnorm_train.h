/*
 * rmsnorm_train.h -- C ABI of the GB300 (sm_103a) RMSNorm-for-training library.
 *
 * The operation (flashinfer PR #8827 "fix(cake_rmsnorm): sm_100a and sm_107a dw-accuracy
 * backward routes", description, and its Measurement section's workload line):
 *
 *   forward   rstd = 1 / sqrt(mean_j(x_j^2) + eps)        FP32, one per normalized row
 *             y_j  = BF16(x_j * rstd * w_j)                BF16, round to nearest even
 *             residual form: x := h = BF16(x_in + residual), and h is written too
 *   backward  xhat = x * rstd,  g = dy * w,  c = mean_j(g_j * xhat_j)
 *             dx_j = BF16(rstd * (g_j - xhat_j * c) [+ dh_j])
 *             dw_j = sum over all normalized rows of dy_j * xhat_j   (FP32)
 *
 * Two backward modes share one forward: deterministic != 0 gives bit-identical dw run to
 * run and across GPUs of any SM count (the row -> partial mapping depends on T, nh, H and
 * whether dh is given, never on the GPU; a second kernel adds the partials in a fixed
 * order); deterministic == 0 gives each CTA a fixed prefix of rows and hands the last
 * rows out to the CTAs as they free up (no CTA idles while another still has a queue of
 * rows), so a CTA's dw partial covers rows that vary from run to run and dw may differ
 * between runs in its last bits (both modes keep dw within the same budget); where a CTA
 * would own fewer than eight ring depths of rows it takes the deterministic partition
 * instead (too few rows for the hand-out to even the CTAs out).  dx is the same in both
 * modes, bit for bit.
 *
 * Rows and views (same PR, description: per-head views [T,24,256] strided and [T,4,256]
 * contiguous with a shared w[256]).  A normalized row is a pair (token t, head h),
 * r = t*nh + h, with H elements; plain rows are nh = 1.  The forward's input activation
 * (x / x_in / residual) and the backward's saved input are read through element strides:
 * row r starts at element t*s_tok + h*s_head.  Every other tensor is contiguous:
 * y, h_out, dy, dh, dx are [T, nh, H]; rstd is [T, nh]; w and dw are [H].
 *
 * Conventions common to every entry point:
 *  - Pointers are DEVICE pointers on the current CUDA device, except where a comment says
 *    otherwise.  BF16 = IEEE bfloat16 bit patterns (uint16 storage).
 *  - Ownership: the caller owns every buffer, the workspace included.  The library never
 *    allocates, frees or synchronizes; all work is enqueued on `stream` (a cudaStream_t
 *    passed as void*; NULL = the legacy default stream) and is asynchronous.
 *  - Alignment: every tensor pointer 16-byte aligned, except rstd (4-byte aligned; the
 *    backward reads it fastest when it is 16-byte aligned); H a multiple of 8; s_tok and
 *    s_head multiples of 8 elements (each row is a 16-byte-aligned run).
 *  - Limits: 8 <= H <= 8192, T >= 0, nh >= 1, T*nh <= 2^31 - 2^16.
 *  - Outputs must not overlap inputs.
 *  - Errors: argument checks happen before anything is enqueued and return a nonzero
 *    status without touching memory; RMSN_ERR_CUDA reports a failed launch (the CUDA
 *    error is left for cudaGetLastError()).  rmsnorm_train_status_str names a status.
 */
#ifndef RMSNORM_TRAIN_H
#define RMSNORM_TRAIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RMSN_OK 0
#define RMSN_ERR_INVALID_ARG 1 /* null/misaligned pointer, bad size, stride or dtype */
#define RMSN_ERR_UNSUPPORTED 2 /* H above 8192 or T*nh too large */
#define RMSN_ERR_WORKSPACE 3   /* workspace missing or smaller than required */
#define RMSN_ERR_CUDA 4        /* a CUDA runtime call or launch failed */
#define RMSN_ERR_DEVICE 5      /* current device is not compute capability 10.3 */
#define RMSN_ERR_SCRATCH_LIMIT 6 /* rmsnorm_train_bwd_noalloc: shape exceeds its scratch */

#define RMSN_W_BF16 0 /* w is BF16 [H] */
#define RMSN_W_FP32 1 /* w is FP32 [H] */

/*
 * Forward: y (BF16) and rstd (FP32); with `residual` != NULL also h_out = BF16(x + residual)
 * and the norm is taken of h_out.  (PR #8827 description: the forward's outputs, and the
 * fused residual add at H6144; the workload line: eps 1e-6, y / h_new BF16, rstd FP32.)
 *
 *   x         BF16, read through (s_tok, s_head): the activation (x_in in residual form)
 *   residual  BF16 or NULL, same strides as x
 *   w         [H], dtype w_dtype (RMSN_W_BF16 or RMSN_W_FP32)
 *   y         BF16 [T, nh, H] out
 *   h_out     BF16 [T, nh, H] out; required iff residual != NULL, else must be NULL
 *   rstd      FP32 [T, nh] out
 *   eps       added to mean(x^2) inside the square root; finite, >= 0
 * T*nh == 0 returns RMSN_OK with nothing enqueued.
 */
int rmsnorm_train_fwd(const void* x, const void* residual, const void* w, int w_dtype,
                      void* y, void* h_out, float* rstd,
                      int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
                      float eps, void* stream);

/*
 * Bytes of device workspace rmsnorm_train_bwd needs for this shape and mode: 0 for
 * T*nh <= 256 rows (done in one launch without a workspace) and for T*nh == 0.  Above
 * that, P partials of 2*H floats (P <= 152 per CTA an SM the launch shape keeps
 * resident, a function of (T, nh, H) only), and for deterministic == 0 a 16-byte row
 * counter slot before them.  Returns 0 on invalid sizes.  Host-only computation: no
 * device access.
 */
size_t rmsnorm_train_bwd_workspace_bytes(int64_t T, int32_t nh, int32_t H, int deterministic);

/*
 * Backward: dx (BF16) and dw (FP32).  (PR #8827 description: the backward's outputs and
 * the two modes; PR #8849 and the route notes of PR #8827: dw must stay within per-element
 * atol 1e-4 + rtol 1e-4 of an FP64 sum, which this library meets with compensated FP32
 * per-partition sums and a fixed-order compensated finish.)
 *
 *   x          BF16, the forward's normalized input (x, or h_out of the residual form),
 *              read through (s_tok, s_head)
 *   dy         BF16 [T, nh, H], upstream gradient of y
 *   dh         BF16 [T, nh, H] or NULL: upstream gradient of h_out in the residual form,
 *              added to dx (the combined gradient of x_in and residual)
 *   rstd       FP32 [T, nh] as returned by the forward
 *   w          [H], dtype w_dtype
 *   dx         BF16 [T, nh, H] out
 *   dw         FP32 [H] out, overwritten (not accumulated); zero-filled when T*nh == 0
 *   workspace  device scratch of >= rmsnorm_train_bwd_workspace_bytes(...) bytes,
 *              16-byte aligned, no initial contents required (the non-deterministic
 *              mode's row counter is opened by each call, under a per-call tag); clobbered
 *              by the call (may be NULL when that size is 0).  Two calls that may overlap
 *              on the GPU need separate workspaces.
 *   deterministic  0 or 1 (see the top of this file)
 */
int rmsnorm_train_bwd(const void* x, const void* dy, const void* dh, const float* rstd,
                      const void* w, int w_dtype, void* dx, float* dw,
                      void* workspace, size_t workspace_bytes,
                      int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
                      int deterministic, void* stream);

/*
 * Backward that is not handed rstd: it recomputes rstd = 1/sqrt(mean(x^2) + eps) from the
 * rows it already reads (one more multiply-add an element, no extra pass over x) and
 * writes it to rstd_out.  For steps that checkpoint the forward's input but not its
 * statistics: flashinfer PR #8827's Measurement section times the checkpointed step
 * (forward, forward again, backward) as an op of its own, and this entry point replaces
 * the second forward when only the backward needs it.
 *
 * Arguments as rmsnorm_train_bwd, except:
 *   rstd_out   FP32 [T, nh] out (required, 4-byte aligned): the recomputed rstd, the
 *              forward's formula in FP32 (its sum of squares may add in another order, so
 *              a bit may differ from the forward's; both stay within 1e-6 of the exact
 *              value)
 *   eps        as passed to the forward; finite, >= 0
 * The workspace is rmsnorm_train_bwd_workspace_bytes(T, nh, H, deterministic) bytes.  dx
 * and dw follow the rules of rmsnorm_train_bwd with the recomputed rstd; the determinism
 * contract is the same.
 */
int rmsnorm_train_bwd_recompute(const void* x, const void* dy, const void* dh, const void* w,
                                int w_dtype, void* dx, float* dw, float* rstd_out,
                                void* workspace, size_t workspace_bytes, int64_t T, int32_t nh,
                                int32_t H, int64_t s_tok, int64_t s_head, float eps,
                                int deterministic, void* stream);

/*
 * Backward for callers that cannot allocate device memory where they call it -- e.g. a
 * plugin's enqueue callback in a runtime that forbids allocation there, or a host with no
 * device allocator to provide a workspace.  (The pages have no counterpart: this entry
 * point exists for such callers only.)  Same arguments, results and modes as
 * rmsnorm_train_bwd minus the workspace: the dw partials live in a 16 MiB array of device
 * memory built into the library, which each device that loads the library holds until
 * the process exits.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on a device looks up that array's device address (a runtime call,
 *    no allocation); make that first call before capturing a stream into a graph.
 *  - Every call on a device shares the array; calls that may overlap on the GPU (e.g. on
 *    two unordered streams) race on it and must be serialized by the caller.  No initial
 *    contents are needed.
 *  - Returns RMSN_ERR_SCRATCH_LIMIT, with nothing enqueued, when the shape needs more than
 *    16 MiB (rmsnorm_train_bwd_workspace_bytes() > 16 MiB).  No supported shape does:
 *    either mode needs at most 16 + 152 x 2 x 8192 x 4 bytes (9.5 MiB), so this status
 *    is a guard, not a case a caller meets.
 */
int rmsnorm_train_bwd_noalloc(const void* x, const void* dy, const void* dh, const float* rstd,
                              const void* w, int w_dtype, void* dx, float* dw,
                              int64_t T, int32_t nh, int32_t H, int64_t s_tok, int64_t s_head,
                              int deterministic, void* stream);

/*
 * The launch plan the library uses for one op at width H: for tests and diagnostics.
 * No device access; the result depends on H and op only.
 *   op     RMSN_PLAN_FWD, RMSN_PLAN_FWD_RESIDUAL, RMSN_PLAN_BWD or RMSN_PLAN_BWD_DH (the
 *          deterministic backward without / with dh), RMSN_PLAN_BWD_ND or
 *          RMSN_PLAN_BWD_ND_DH (the non-deterministic backward: the same plans, as both
 *          modes run one row-pass program on one launch shape)
 *   out    host array receiving min(n_out, RMSN_PLAN_FIELDS) values, in this order:
 *            [0] 16-byte column vectors (8 columns) per consumer thread
 *            [1] threads per row group (8 or 16: sub-warp groups; else whole warps)
 *            [2] row groups per CTA (= rows per ring stage)
 *            [3] ring stages
 *            [4] threads per CTA (the row groups + one producer warp)
 *            [5] dynamic shared memory bytes per CTA
 *            [6] shape class (forward: 0 two CTAs an SM, 1 one CTA an SM; backward:
 *                0 narrow, 1 several row groups, 2 wide, 3 several row groups with the dw
 *                sums in tensor memory)
 *            [7] most threads a CTA of that class's kernel build may have
 *            [8] CTAs per SM that class's kernel build is made for
 * Returns RMSN_OK; RMSN_ERR_INVALID_ARG for an unknown op, out == NULL, n_out < 0 or H
 * not a positive multiple of 8; RMSN_ERR_UNSUPPORTED for H above 8192.
 */
#define RMSN_PLAN_FWD 0
#define RMSN_PLAN_FWD_RESIDUAL 1
#define RMSN_PLAN_BWD 2
#define RMSN_PLAN_BWD_DH 3
#define RMSN_PLAN_BWD_ND 4
#define RMSN_PLAN_BWD_ND_DH 5
#define RMSN_PLAN_FIELDS 9
int rmsnorm_train_launch_plan(int32_t H, int op, int64_t* out, int n_out);

/* Static string naming a status code (never NULL). */
const char* rmsnorm_train_status_str(int status);

/*
 * Reads (and, if reset != 0, clears) the library's device-side error word on the current
 * device into *flags (host pointer).  Nonzero means a kernel gave up on a bounded wait
 * (bit 0: a consumer waited too long for staged data or for a row's reduction; bit 1:
 * the staging producer waited too long for a free buffer); that call's outputs are then
 * unspecified.  This entry point
 * SYNCHRONIZES the device; it is meant for tests and diagnostics, not the hot path.
 */
int rmsnorm_train_device_error(unsigned int* flags, int reset);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_TRAIN_H */
