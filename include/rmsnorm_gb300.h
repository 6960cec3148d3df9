/*
 * rmsnorm_gb300.h -- C ABI of the GB300 (sm_103a) RMSNorm library (with
 * LayerNorm alongside).
 *
 * What it computes (FlyDSL pages):
 *   forward, per row m of an [M,N] input:
 *       rstd_m = 1 / sqrt(mean_j x_mj^2 + eps),   y_mj = x_mj * rstd_m * gamma_j
 *     -- issue #769 "Add rmsnorm backward (+ forward saves rstd)", section
 *        "Current state" (the per-row rrms), and PR #800's commit message
 *        "Makes RMSNorm training-capable" (rstd is 1/RMS, fp32, shape (M,)).
 *   backward, per row, with x_hat = x * rstd and wdy = dy * gamma:
 *       c1 = mean_j(x_hat_j * wdy_j),  dx_j = (wdy_j - x_hat_j * c1) * rstd
 *     and over all rows  dweight_j = sum_m dy_mj * x_hat_mj  (fp32, length N)
 *     -- issue #769, section "Math (matches quack rmsnorm_bwd_ref)".
 *   fused-add (prenorm): added = x + residual is saved (residual_out); the
 *     backward runs on `added`, adds dresidual_out (if given) to dx, and dx is
 *     also the gradient of residual (dx == dresidual)
 *     -- PR #800 "Add fused-add / residual backward", section "What's included".
 *
 * Conventions shared by every call:
 *   - All [M,N] tensors are row-major and contiguous (row stride N elements);
 *     gamma, dweight are [N]; rstd is fp32 [M]; dweight_f32 is fp32 [N].
 *   - One I/O dtype per call (rn_dtype) for x / residual / added / gamma /
 *     dy / dresidual_out / y / out / residual_out / dx / dweight: the kernels
 *     read every operand with that one element type. Every reduction and the
 *     weight-gradient accumulation run in fp32; outputs are rounded to the
 *     I/O dtype once, to nearest even.
 *   - Pointers are DEVICE pointers on the calling thread's current CUDA
 *     device; the caller owns every buffer. Nothing is allocated or freed.
 *     Each buffer starts at a multiple of its element size (the I/O dtype's;
 *     4 bytes for the fp32 ones), else RN_ERR_INVALID_ARG. Any further
 *     alignment is optional: 16-byte aligned row tensors with 16-byte
 *     multiple rows take the fastest engines.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *     asynchronous: they enqueue kernels on `stream` and return.
 *   - Errors: argument checks run before anything is enqueued and return
 *     RN_ERR_INVALID_ARG / RN_ERR_UNSUPPORTED / RN_ERR_WORKSPACE with nothing
 *     launched; a failed launch returns RN_ERR_CUDA. rn_last_error() gives a
 *     message for the calling thread's last failure.
 *   - Output buffers must not overlap any input, except that the backward's
 *     dx may be the very same buffer as dresidual_out (each element is read
 *     before it is overwritten).
 *   - N >= 1; M >= 0. M == 0 is a valid empty batch (the backward then writes
 *     a zero dweight).
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rn_dtype { RN_F32 = 0, RN_F16 = 1, RN_BF16 = 2 } rn_dtype;

typedef enum rn_status {
    RN_OK = 0,
    RN_ERR_INVALID_ARG = 1,  /* null pointer, a buffer not aligned to its element size,
                                bad size, bad dtype code, bad option */
    RN_ERR_UNSUPPORTED = 2,  /* shape/alignment no engine handles (e.g. N too large) */
    RN_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    RN_ERR_WORKSPACE = 4     /* workspace missing, misaligned or too small */
} rn_status;

/* Version of this ABI (increments on any incompatible change). */
int rn_abi_version(void);

/* Static text for a status code. */
const char *rn_status_string(int status);

/* Message describing the calling thread's most recent failure ("" if none). */
const char *rn_last_error(void);

/*
 * Forward, plain RMSNorm (issue #769 "Current state"; PR #800 commit
 * "Makes RMSNorm training-capable", store_rstd).
 *   x      [M,N] dtype, in
 *   gamma  [N]   dtype, in
 *   eps    added to the mean square before the reciprocal square root
 *   y      [M,N] dtype, out: x * rstd * gamma
 *   rstd   [M] fp32, out, may be NULL (then not stored)
 */
rn_status rn_rmsnorm_fwd(const void *x, const void *gamma, float eps, void *y, float *rstd,
                         int64_t M, int64_t N, int dtype, void *stream);

/*
 * Forward, fused-add (prenorm) RMSNorm (PR #800 "What's included").
 *   x, residual   [M,N] dtype, in
 *   gamma         [N] dtype, in
 *   out           [M,N] dtype, out: added * rstd * gamma
 *   residual_out  [M,N] dtype, out: added = x + residual, rounded to dtype;
 *                 the statistic and `out` are computed from this rounded value
 *   rstd          [M] fp32, out (of `added`), may be NULL
 */
rn_status rn_fused_add_rmsnorm_fwd(const void *x, const void *residual, const void *gamma,
                                   float eps, void *out, void *residual_out, float *rstd,
                                   int64_t M, int64_t N, int dtype, void *stream);

/*
 * Bytes of workspace the backward needs on the current device for an [M,N]
 * problem: a 256-byte header plus up to two fp32 rows of N per SM (the
 * per-CTA partials of the weight gradient). Needs a CUDA device; writes
 * *bytes. The workspace must be 256-byte aligned; its contents need no
 * initialisation and are scratch between calls. Calls that share one
 * workspace must be ordered on the GPU (one stream, or events).
 */
rn_status rn_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes);

/*
 * Backward, plain RMSNorm (issue #769 "Math").
 *   x            [M,N] dtype, in (the forward's input)
 *   gamma        [N] dtype, in
 *   dy           [M,N] dtype, in (gradient of y)
 *   rstd         [M] fp32, in: the statistic the forward saved (not recomputed)
 *   dx           [M,N] dtype, out
 *   dweight_f32  [N] fp32, out, may be NULL: fully overwritten with
 *                sum_m dy*x_hat
 *   dweight      [N] dtype, out, may be NULL: that sum rounded to dtype
 *   workspace    device buffer of >= rn_bwd_workspace_bytes(M,N,dtype) bytes
 * Every step (zero, row pass, cross-row reduction, cast) runs inside this call.
 * Without dweight_f32 the fp32 sum is not stored and the weight gradient takes
 * the deterministic scratch mode (per-CTA partial rows in the workspace, then
 * one kernel that sums them in a fixed order and writes dweight): one launch
 * fewer than the atomic mode's zero, row pass and cast. With neither
 * dweight_f32 nor dweight no weight gradient is produced (the row pass alone).
 */
rn_status rn_rmsnorm_bwd(const void *x, const void *gamma, const void *dy, const float *rstd,
                         void *dx, float *dweight_f32, void *dweight,
                         void *workspace, size_t workspace_bytes,
                         int64_t M, int64_t N, int dtype, void *stream);

/*
 * Backward, fused-add RMSNorm (PR #800 "What's included").
 *   added          [M,N] dtype, in: the saved x + residual (residual_out)
 *   gamma, dy, rstd as for rn_rmsnorm_bwd (rstd is the statistic of `added`)
 *   dresidual_out  [M,N] dtype, in, may be NULL (read as zeros): gradient
 *                  flowing into residual_out
 *   dx             [M,N] dtype, out: (wdy - a_hat*c1)*rstd + dresidual_out;
 *                  it is both the x gradient and the residual gradient. It may
 *                  be the same buffer as dresidual_out.
 *   dweight_f32, dweight, workspace as for rn_rmsnorm_bwd.
 */
rn_status rn_fused_add_rmsnorm_bwd(const void *added, const void *gamma, const void *dy,
                                   const float *rstd, const void *dresidual_out, void *dx,
                                   float *dweight_f32, void *dweight,
                                   void *workspace, size_t workspace_bytes,
                                   int64_t M, int64_t N, int dtype, void *stream);

/*
 * LayerNorm. The FlyDSL pages plan its backward as the RMSNorm backward with
 * mean handling and a bias gradient added, over a forward that saves the
 * per-row mean and rstd (issue #769, plan item 6 "layernorm backward -- same
 * pattern" and "PR 5 -- LayerNorm backward": "adding mean handling + dbias").
 * The formulas are the textbook definition:
 *   forward, per row:  mean = (1/N) sum_j x_j,  var = (1/N) sum_j (x_j - mean)^2,
 *                      rstd = 1/sqrt(var + eps),
 *                      y_j = (x_j - mean) * rstd * gamma_j + beta_j
 *   backward, per row with x_hat = (x - mean)*rstd and wdy = dy*gamma:
 *                      c1 = mean_j(x_hat_j*wdy_j),  c2 = mean_j(wdy_j),
 *                      dx_j = (wdy_j - c2 - x_hat_j*c1) * rstd
 *   over all rows:     dgamma_j = sum_m dy_mj*x_hat_mj,  dbeta_j = sum_m dy_mj
 * The conventions above apply (one I/O dtype; device pointers; fp32 math).
 */

/*
 * Forward, LayerNorm.
 *   x      [M,N] dtype, in
 *   gamma  [N] dtype, in
 *   beta   [N] dtype, in, may be NULL (no bias)
 *   eps    added to the variance before the reciprocal square root
 *   y      [M,N] dtype, out
 *   mean   [M] fp32, out, may be NULL (then not stored)
 *   rstd   [M] fp32, out, may be NULL (then not stored)
 */
rn_status rn_layernorm_fwd(const void *x, const void *gamma, const void *beta, float eps, void *y,
                           float *mean, float *rstd, int64_t M, int64_t N, int dtype,
                           void *stream);

/*
 * Bytes of workspace rn_layernorm_bwd needs on the current device: a 256-byte
 * header plus up to two fp32 rows of 2N per SM (per-CTA partials of dgamma
 * and dbeta side by side). Same rules as rn_bwd_workspace_bytes.
 */
rn_status rn_layernorm_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes);

/*
 * Backward, LayerNorm.
 *   x           [M,N] dtype, in (the forward's input)
 *   gamma       [N] dtype, in
 *   dy          [M,N] dtype, in (gradient of y)
 *   mean, rstd  [M] fp32, in: the statistics the forward saved (not recomputed)
 *   dx          [M,N] dtype, out; must not overlap any input
 *   dgamma_f32  [N] fp32, out, may be NULL: fully overwritten with sum_m dy*x_hat
 *   dbeta_f32   [N] fp32, out, may be NULL: sum_m dy; must not overlap
 *               dgamma_f32
 *   dgamma      [N] dtype, out, may be NULL: the dgamma sum rounded to dtype
 *   dbeta       [N] dtype, out, may be NULL: the dbeta sum rounded to dtype
 *   workspace   >= rn_layernorm_bwd_workspace_bytes(M,N,dtype) bytes
 * Every step (zero, row pass, cross-row reduction, casts) runs inside this
 * call; RN_OPT_* options apply as for the RMSNorm backward. The atomic mode
 * needs the fp32 buffer of every gradient asked for (dgamma_f32, and
 * dbeta_f32 when dbeta is asked for); otherwise the deterministic scratch mode
 * runs, as for rn_rmsnorm_bwd without dweight_f32. Gradients whose two
 * buffers are both NULL are not produced (dbeta: no bias).
 */
rn_status rn_layernorm_bwd(const void *x, const void *gamma, const void *dy, const float *mean,
                           const float *rstd, void *dx, float *dgamma_f32, float *dbeta_f32,
                           void *dgamma, void *dbeta, void *workspace, size_t workspace_bytes,
                           int64_t M, int64_t N, int dtype, void *stream);

/*
 * Backward, plain RMSNorm, without a caller workspace. (This call has no
 * counterpart on the FlyDSL pages; it exists for callers that cannot
 * allocate device memory when they run the backward -- e.g. code running
 * while a caching allocator or memory pool is locked or being torn down, or
 * an embedder that fixes every device allocation up front.)
 *   Arguments, layouts, outputs and results are those of rn_rmsnorm_bwd.
 *   The scratch comes from a fixed 16 MiB array inside the library's device
 *   image, held by every GPU that loads the library until the process exits.
 *   Problems needing more scratch than that (rn_bwd_workspace_bytes(M, N,
 *   dtype) > 16 MiB, i.e. N above ~13,800 on a 152-SM GB300) are refused
 *   with RN_ERR_UNSUPPORTED and a message in rn_last_error(); nothing is
 *   launched. The call allocates nothing and frees nothing.
 *   The first call on a device looks up the array's device address on that
 *   device (cudaGetSymbolAddress) and keeps it for the life of the process;
 *   make that first call before any stream capture. A device reset
 *   (cudaDeviceReset) while this library is loaded is not supported: it
 *   reloads the device image, and the kept address would then be stale. All
 *   calls share the one array: nothing in it needs to start at
 *   zero (every call overwrites the part it reads), but calls that could run
 *   at the same time on the GPU (different streams without ordering) race on
 *   it and give wrong results. Order such calls on one stream or with events.
 */
rn_status rn_rmsnorm_bwd_noalloc(const void *x, const void *gamma, const void *dy,
                                 const float *rstd, void *dx, float *dweight_f32, void *dweight,
                                 int64_t M, int64_t N, int dtype, void *stream);

/*
 * Tuning / test options. They are process-wide, not thread-safe, and apply
 * to calls made after they are set; value 0 always means "automatic".
 */
typedef enum rn_option {
    RN_OPT_BWD_ENGINE = 0,    /* 1 = row engine (async-copy ring), 2 = generic engines (the
                                 default for rows that are not 16-byte multiples or bases off
                                 16 bytes; which one runs depends on the row size and on whether
                                 the row tensors share one alignment phase: the staged
                                 phase-class kernel up to 2048 whole 16-byte chunks, vector
                                 kernel past that, element-wise kernel for mixed phases),
                                 3 = cluster engine (RMSNorm backward: a row split across a
                                 thread-block cluster; chosen by default for aligned rows of
                                 more than 2048 16-byte chunks) */
    RN_OPT_DWEIGHT_MODE = 1,  /* 1 = scratch partials + finalize (deterministic dweight),
                                 2 = fp32 atomics + cast (summation order varies from call to
                                 call). Automatic: scratch when a row tensor holds at most
                                 2 MiB (fewer launches), else atomics where possible */
    RN_OPT_CHUNKS_PER_THREAD = 2, /* row engine and staged phase-class kernels: 16-byte chunks
                                 per thread per row: 1, 2, 4 (default: by row length) */
    RN_OPT_TEAMS_PER_CTA = 3, /* row engine and staged phase-class kernels: rows processed at
                                 once per CTA (1..15; the staged kernels otherwise run a tile of
                                 two teams of 192-256 threads as one team a CTA at two CTAs an
                                 SM); RMSNorm backward phase-class kernel: rows per CTA
                                 iteration (1 or 2) */
    RN_OPT_STAGES = 4,        /* row engine: rows in flight per team (2..8); staged
                                 phase-class kernel: shared-memory slots per team (2..4) */
    RN_OPT_GRID = 5,          /* CTAs of the row pass (default: one per SM; at most 2 per SM) */
    RN_OPT_CLUSTER_SIZE = 6,  /* cluster engine: CTAs per cluster, 2, 4, 8 or 16 */
    RN_OPT_GENERIC_KERNEL = 7, /* backward generic engines: 1 = phase-class kernel (rows held
                                 in registers), 2 = vector kernel, 3 = realigning kernel (RMSNorm,
                                 rows of 16 to 32 KB; taken only when asked for), 4 = element-wise
                                 kernel, 5 = staged phase-class kernel (rows staged in shared
                                 memory by bulk copies; chosen automatically from 2048 rows,
                                 LayerNorm: unless its tile is two teams). A kernel that cannot
                                 take the problem (its row-size range, or tensors at different
                                 alignment phases) falls back to the next one the automatic
                                 choice would make. The forwards on such rows read 5 as "the
                                 staged forward wherever it can run" and any other non-zero
                                 value as "not the staged forward"; their automatic choice
                                 takes the staged forward from 2048 rows (RMSNorm with at least
                                 6 rows a team, fused-add with one team a CTA, either way also
                                 for rows of at most 256 chunks). */
    RN_OPT_TEST_WAIT_TIMEOUT = 8, /* test hook, staged phase-class kernels (RMSNorm and
                                 LayerNorm backward, the forwards): v > 0 makes the first CTA's
                                 first team leave its row v-1 (counted from 0 among that team's
                                 rows) uncopied, so that the team's bounded wait (250 ms) runs
                                 out. The call then leaves output rows (and the weight
                                 gradients) incomplete and rn_take_device_status() reports
                                 bit 0. */
    RN_OPT_COUNT = 9
} rn_option;

rn_status rn_set_option(int option, int value);
int rn_get_option(int option);

/*
 * Text describing the plan the most recent backward or forward call on this
 * thread used: the engine, and for the row engines the tile shape and grid
 * (for a backward also the weight-gradient mode); "" if none. Forward plans
 * start with the operation ("rmsnorm_fwd", "fused_add_fwd", "layernorm_fwd").
 */
const char *rn_last_plan(void);

/*
 * Device status word of the current device (kernels OR bits into it):
 *   bit 0 = a bounded wait inside a kernel ran out (the staged phase-class
 *           kernels, the RMSNorm and LayerNorm backwards and the forwards, wait
 *           at most 250 ms for a row's bulk copies). The team that waited
 *           stopped: the output rows it had not reached (dx, or y, residual_out
 *           and the statistics) and the weight gradients of that call are not
 *           valid. The CUDA context stays usable.
 * Synchronizes the device, stores the word in *status and clears it.
 * Returns RN_ERR_INVALID_ARG for a NULL status, RN_ERR_CUDA if a CUDA call fails.
 */
rn_status rn_take_device_status(unsigned int *status);

/*
 * Timing hook: while both are non-NULL, every backward call records
 * cudaEvent_t `ev_begin` just before its row-pass kernel and `ev_end` just
 * after it, on the call's stream. Pass NULLs to switch off.
 */
rn_status rn_set_profile_events(void *ev_begin, void *ev_end);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
