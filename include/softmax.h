/*
 * softmax.h -- C ABI of libosd_softmax.so: row-wise safe softmax on one GB300
 * (sm_103a) GPU.
 *
 * The operation (every entry point below computes it, or reports on it):
 *
 *     for each row r of a contiguous row-major [rows, cols] array x:
 *         m    = max_j x[r, j]
 *         d    = sum_j exp(x[r, j] - m)
 *         y[r, j] = exp(x[r, j] - m) / d
 *
 * defined in "[CUDA] safe online softmax" (wingedge777.com), section 1 "safe
 * online softmax" (the safe_softmax form: max, exp of the shifted values,
 * divide by their sum), and in the HIP softmax tutorial (forum.sourcefind.cn),
 * section 1 "Softmax operator definition", whose worked example maps
 * [[1,2,3],[1,1,1]] to [[0.0900,0.2447,0.6652],[0.3333,0.3333,0.3333]].
 * The max and the sum are accumulated in fp32 whatever the storage dtype
 * ("Softmax on DCU: from 2.34 ms to 0.62 ms" (czchanglian.com), section 4.5:
 * fp16 storage, fp32 accumulation), and y is rounded to nearest-even into the
 * dtype of x.  Accuracy against the exact (binary64) result y*:
 *     fp32        |y - y*| <= 2e-6 * y* + 2^-126
 *     fp16, bf16  at most 1 ulp from y* rounded to the dtype
 * with no inf or NaN for finite inputs.  Non-finite inputs propagate as IEEE
 * arithmetic does: a NaN or +inf in a row, or a row of all -inf, gives a NaN
 * row; -inf entries in an otherwise finite row give 0.
 *
 * Conventions shared by every entry point:
 *   - x and y are DEVICE pointers to contiguous row-major [rows, cols] arrays
 *     of the same dtype (row stride = cols elements).  The caller owns both;
 *     the library never allocates, frees or copies between host and device.
 *     Pointers must be aligned to the element size (4 bytes for fp32, 2 for
 *     fp16 / bf16); 16-byte aligned rows take the vectorised fast path, any
 *     other alignment is handled by peeling partial 16-byte chunks.
 *   - y may be x itself (in place: every element is read before it is
 *     overwritten); any other overlap of x and y is refused.
 *   - work is enqueued on `stream` (NULL = the legacy default stream) and the
 *     call returns without synchronising.  Faults during execution surface at
 *     the caller's next synchronisation, as for any CUDA launch.
 *   - the current CUDA device is used; per-device attributes (SM count, shared
 *     memory limit, cluster support) are read once per device and cached
 *     (thread-safe).
 *   - return value: SOFTMAX_OK (0) or a negative softmax_status.  Nothing
 *     prints, throws or exits.
 */
#ifndef OSD_SOFTMAX_H
#define OSD_SOFTMAX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *softmax_stream_t;

/* Storage dtype of x and y. */
typedef enum {
    SOFTMAX_F32 = 0,
    SOFTMAX_F16 = 1,
    SOFTMAX_BF16 = 2
} softmax_dtype;

typedef enum {
    SOFTMAX_OK = 0,
    SOFTMAX_ERR_INVALID_ARG = -1,       /* null pointer with non-zero size, rows or cols < 0,
                                           rows*cols*size overflows int64, misaligned pointer,
                                           bad variant id, null out-pointer */
    SOFTMAX_ERR_UNSUPPORTED_DTYPE = -2, /* dtype not in softmax_dtype */
    SOFTMAX_ERR_ALIAS = -3,             /* buffers overlap (other than an allowed in-place call) */
    SOFTMAX_ERR_CUDA = -4,              /* a CUDA runtime call failed; see softmax_last_cuda_error */
    SOFTMAX_ERR_UNSUPPORTED_SHAPE = -5, /* a forced variant cannot serve this shape / device */
    SOFTMAX_ERR_DEVICE_TIMEOUT = -6     /* a bounded device-side wait gave up (see
                                           softmax_get_device_error) */
} softmax_status;

/* Kernel variants the dispatcher chooses among. */
typedef enum {
    SOFTMAX_VARIANT_AUTO = 0,      /* let the dispatcher choose */
    SOFTMAX_VARIANT_ROWGROUP = 1,  /* G = 1..32 lanes per row, row cached in registers */
    SOFTMAX_VARIANT_BLOCK = 2,     /* one CTA per row, row cached in registers (rows of up to
                                      8192 chunks of 16 bytes; past 4096, one CTA per SM
                                      looping over rows) */
    SOFTMAX_VARIANT_BLOCK_TMA = 3, /* persistent CTAs, rows staged in shared memory by bulk
                                      async copies (TMA engine), one HBM read per element */
    SOFTMAX_VARIANT_STREAM = 4,    /* one CTA per row, online (m, d) pass then a re-read pass;
                                      any cols */
    SOFTMAX_VARIANT_SPLITK = 5,    /* a thread-block cluster per row; partial (m, d) merged
                                      through distributed shared memory (one CTA per row when
                                      there are at least as many rows as SMs) */
    SOFTMAX_VARIANT_SPLITK_WIDE = 6, /* P CTAs per row over all SMs, partials merged through a
                                        global workspace in a second launch (softmax_fwd_ws
                                        only: it needs the workspace) */
    SOFTMAX_VARIANT_SPLITK_GRID = 7, /* P CTAs per row over all SMs in one cooperative launch,
                                        partials exchanged at a bounded per-row grid barrier
                                        through library-owned scratch.  Ring form (stages >= 1):
                                        grid_y groups of grid_x CTAs, one CTA per SM, a group
                                        takes every grid_y-th row in turn, each CTA's share of
                                        a row held in one of `stages` shared-memory buffers (one
                                        HBM read); pipelined form (lanes_per_row > 0): grid_y =
                                        1, every CTA on every row, the rows in turn through the
                                        buffers, a fold team of lanes_per_row threads working on
                                        one row while the rest of the CTA writes the row before;
                                        streaming form (stages 0): grid_y = rows */
    SOFTMAX_VARIANT_COUNT = 8
} softmax_variant;

/*
 * softmax_fwd -- y = softmax(x) along the last dimension.
 *   x      device pointer, [rows, cols] of `dtype`, read only.
 *   y      device pointer, [rows, cols] of `dtype`, written in full.
 *   rows   number of rows (>= 0).  rows == 0 or cols == 0: SOFTMAX_OK, no launch.
 *   cols   row length (>= 0).  cols == 1 gives y = 1.
 *   dtype  softmax_dtype.
 *   stream CUDA stream the work is enqueued on.
 * Chooses a kernel from cols * sizeof(dtype), rows, the SM count and the
 * 16-byte alignment of x, y and the row stride (the cols-based dispatch of the
 * HIP softmax tutorial, section 7, rebuilt for this GPU), then issues exactly
 * one kernel launch.
 */
int softmax_fwd(const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                softmax_stream_t stream);

/*
 * softmax_fwd_variant -- as softmax_fwd, with the kernel forced (for tests and
 * benchmarks).  variant = SOFTMAX_VARIANT_AUTO behaves exactly like
 * softmax_fwd.  Returns SOFTMAX_ERR_UNSUPPORTED_SHAPE when the forced variant
 * cannot serve the shape on this device (e.g. a row too long to cache on
 * chip for ROWGROUP / BLOCK / BLOCK_TMA, or no cluster launch for SPLITK).
 */
int softmax_fwd_variant(const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                        int variant, softmax_stream_t stream);

/*
 * softmax_fwd_masked -- scaled, masked softmax for attention scores:
 *     z[r, j] = scale * x[r, j] + mask[r % mask_rows, j]        (mask optional)
 *     with causal_q > 0:  z[r, j] = -inf for j > i + (cols - causal_q),
 *                         i = r % causal_q (query blocks of causal_q rows whose
 *                         last query sees every key)
 *     y[r, :] = softmax(z[r, :])
 * The scale and the masks are applied as x is loaded; the logits never go to
 * memory ("Softmax on DCU", section 9: fuse the scale and the mask into the
 * softmax for attention; the Pangu-Weather profile, section 6, tried a bias +
 * mask + softmax fusion).  For attention scores [B, H, Sq, Sk]: rows = B*H*Sq,
 * cols = Sk, scale = 1/sqrt(head dim), causal_q = Sq; a key-padding mask is
 * [1, Sk] (mask_rows = 1), a per-query mask [Sq, Sk] (mask_rows = Sq).
 *   mask       device pointer, [mask_rows, cols] of `dtype`, or NULL.  It may
 *              overlap x (both are only read), not y (SOFTMAX_ERR_ALIAS).
 *   mask_rows  >= 1 when mask is given (ignored otherwise).
 *   causal_q   0 (no causal cut) or the query block length.  A row with no
 *              visible key is all -inf and comes out NaN, as the definition
 *              gives.
 * Accuracy: as softmax_fwd (fp32 2e-6 relative; fp16 / bf16 within 1 ulp of
 * the correctly rounded result) against the exact softmax of z formed from
 * the float `scale` as passed, whatever the size of the logits: fp32 carries
 * z as a two-float pair; fp16 / bf16 form z - max with a rounding relative to
 * z - max itself wherever the row's largest logit reaches 512 in magnitude
 * (below that one fp32 FMA for z is accurate enough).
 * Rows up to 2048 chunks of 16 bytes (32 KiB: 16384 fp16 / bf16 or 8192 fp32
 * keys): SOFTMAX_ERR_UNSUPPORTED_SHAPE beyond.  Alignment, streams, errors:
 * as softmax_fwd.
 */
int softmax_fwd_masked(const void *x, void *y, int64_t rows, int64_t cols, int dtype, float scale,
                       const void *mask, int64_t mask_rows, int64_t causal_q, softmax_stream_t stream);

/* softmax_fwd_masked_variant -- softmax_fwd_masked with the kernel forced
 * (ROWGROUP or BLOCK; AUTO = softmax_fwd_masked). */
int softmax_fwd_masked_variant(const void *x, void *y, int64_t rows, int64_t cols, int dtype, float scale,
                               const void *mask, int64_t mask_rows, int64_t causal_q, int variant,
                               softmax_stream_t stream);

/*
 * softmax_bwd -- the backward pass of softmax along the last dimension:
 *     s_r = sum_k dy[r, k] * y[r, k];   dx[r, j] = y[r, j] * (dy[r, j] - s_r)
 * the derivative of the definition above (dy_i/dx_j = y_i (delta_ij - y_j));
 * "Softmax on DCU", section 5.4, names the backward pass as the work that
 * follows the forward one.
 *   y      device pointer, [rows, cols] of `dtype`: the forward output.
 *   dy     device pointer, [rows, cols] of `dtype`: the upstream gradient.
 *   dx     device pointer, [rows, cols] of `dtype`: written in full.
 * s is accumulated in fp32 with compensated (TwoSum) additions; dx is rounded
 * to nearest-even into `dtype`.  Accuracy against the exact result dx*:
 *     |dx - dx*| <= u(dx*) + 8 * 2^-24 * y_j * (|dy_j| + sum_k |dy_k y_k|)
 * with u = 1 ulp of the dtype at dx* for fp16 / bf16 and 2e-6 * |dx*| for
 * fp32; the second term is the fp32 cancellation budget of dy_j - s.
 * y and dy are only read (they may be the same buffer); dx may be exactly y or
 * exactly dy (in place) and must not overlap either otherwise
 * (SOFTMAX_ERR_ALIAS).  Alignment, streams, errors: as softmax_fwd.
 * Kernels: ROWGROUP (rows of up to 128 chunks of 16 bytes), BLOCK (up to 4096),
 * STREAM (any).
 */
int softmax_bwd(const void *y, const void *dy, void *dx, int64_t rows, int64_t cols, int dtype,
                softmax_stream_t stream);

/* softmax_bwd_variant -- softmax_bwd with the kernel forced (ROWGROUP, BLOCK or
 * STREAM; AUTO = softmax_bwd); SOFTMAX_ERR_UNSUPPORTED_SHAPE when it cannot
 * serve the shape. */
int softmax_bwd_variant(const void *y, const void *dy, void *dx, int64_t rows, int64_t cols, int dtype,
                        int variant, softmax_stream_t stream);

/*
 * softmax_fwd_ws -- softmax_fwd with a caller-provided device workspace, which
 * lets few, very long rows use every SM: each row is split over P CTAs (about
 * two CTAs per SM over all rows) whose partial statistics are written to the
 * workspace by a first launch and merged by every CTA of the row in a second
 * launch that also writes y (SPLITK_WIDE; the split of "[CUDA] safe online
 * softmax", section 3.2, with the caller owning the partials' memory).  For
 * shapes that do not need it, or when workspace_bytes is smaller than
 * softmax_workspace_size reports, it behaves exactly like softmax_fwd.
 *   workspace        device pointer, 16-byte aligned, not overlapping x or y;
 *                    NULL only with workspace_bytes == 0.  Its contents on
 *                    entry do not matter; it is scratch until the second
 *                    launch has finished (stream order).  Calls that share a
 *                    workspace must not overlap on the GPU.
 *   workspace_bytes  its size.
 * Returns as softmax_fwd; SOFTMAX_ERR_ALIAS if the workspace overlaps x or y.
 */
int softmax_fwd_ws(const void *x, void *y, int64_t rows, int64_t cols, int dtype, void *workspace,
                   uint64_t workspace_bytes, softmax_stream_t stream);

/*
 * softmax_workspace_size -- bytes of workspace softmax_fwd_ws uses for these
 * arguments on the current device (0 when its choice needs none): rows * P *
 * 16 with P the CTAs per row.  Validates the arguments as softmax_fwd does.
 */
int softmax_workspace_size(const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
                           uint64_t *bytes);

/*
 * softmax_fwd_noalloc -- the SPLITK_WIDE path of softmax_fwd_ws for callers
 * that may not allocate device memory themselves (a plugin whose host engine
 * owns every device allocation and passes it only x and y; a latency-critical
 * path where cudaMalloc, which may synchronise the device, is not allowed).
 * It takes its scratch from a fixed array inside the library instead of a
 * caller workspace and calls no allocating routine.  There is no counterpart
 * on the pages: they allocate their split-k partials per call.
 *   x, y, rows, cols, dtype, stream   as softmax_fwd.
 * Always runs the two-launch wide split: each row is split over P CTAs
 * (about 2 x SMs / rows, at least one 16-byte load step per thread, at most
 * 1024) whose partial statistics go to the array.
 * Limit: rows x P <= 4096 partial slots (the array is 64 KiB, held on every
 * GPU that loads the library until the process exits); larger shapes return
 * SOFTMAX_ERR_UNSUPPORTED_SHAPE.  On a 152-SM GB300 any rows <= 4096 fits.
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  If the lookup fails, the call returns SOFTMAX_ERR_CUDA and the
 * next call on that device looks it up again (only a successful lookup is
 * kept).  Every call shares the array and it keeps the last call's
 * contents; nothing in it needs to start at zero (the first launch writes
 * every slot the second reads).  Calls that overlap on the GPU -- on
 * different streams, or from different host threads -- race on the array and
 * must be serialised by the caller.
 */
int softmax_fwd_noalloc(const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                        softmax_stream_t stream);

/*
 * layernorm_fwd -- LayerNorm along the last dimension, on the softmax's
 * read - reduce - normalise - write skeleton ("Softmax on DCU", section 9,
 * names LayerNorm and RMSNorm as operators of that shape; the Pangu-Weather
 * profile, section 3, standardises fp16 rows with fp32 mean and variance):
 *     mu   = (1/n) sum_j x[r, j]                 n = cols
 *     var  = (1/n) sum_j (x[r, j] - mu)^2        population variance
 *     rstd = 1 / sqrt(var + eps)
 *     y[r, j] = (x[r, j] - mu) * rstd * gamma[j] + beta[j]
 *   x, y    as softmax_fwd (same dtype; y may be x itself, in place).
 *   gamma   device pointer, [cols] of `dtype`, or NULL (gain 1).
 *   beta    device pointer, [cols] of `dtype`, or NULL (bias 0).  Neither may
 *           overlap y.
 *   eps     >= 0 and finite, added to the variance.
 *   mean    device pointer, [rows] fp32, or NULL: mu of each row.
 *   rstd    device pointer, [rows] fp32, or NULL: rstd of each row.  mean and
 *           rstd must be 4-byte aligned and overlap nothing else.
 * The row is held in registers between its reductions (one HBM read of x, one
 * write of y); mu and var are accumulated in fp32 (compensated for fp32
 * input) and var is taken about mu, from the registers; rstd is the SFU's
 * reciprocal square root (about 2 ulp of fp32).  Accuracy against the
 * exact result y*:
 *     |y - y*| <= u(y*) + 64 * 2^-24 * (|gamma_j| * (|z_j| + a * rstd) + |beta_j|)
 * with z_j = (x_j - mu) * rstd, a = (1/n) sum_j |x_j| and u = 1 ulp of the
 * dtype at y* for fp16 / bf16, 0 for fp32 (the second term is the fp32
 * rounding of the statistics); mean and rstd within 64 * 2^-24 of a and of
 * rstd*.  Rows of up to 4096 chunks of 16 bytes (64 KiB):
 * SOFTMAX_ERR_UNSUPPORTED_SHAPE beyond.  Streams, errors: as softmax_fwd.
 */
int layernorm_fwd(const void *x, void *y, int64_t rows, int64_t cols, int dtype, const void *gamma,
                  const void *beta, float eps, float *mean, float *rstd, softmax_stream_t stream);

/*
 * rmsnorm_fwd -- RMSNorm along the last dimension:
 *     rstd = 1 / sqrt((1/n) sum_j x[r, j]^2 + eps);   y[r, j] = x[r, j] * rstd * gamma[j]
 * Arguments, accuracy (without the a * rstd term) and limits as
 * layernorm_fwd, with no bias and no mean.
 */
int rmsnorm_fwd(const void *x, void *y, int64_t rows, int64_t cols, int dtype, const void *gamma, float eps,
                float *rstd, softmax_stream_t stream);

/* norm_fwd_variant -- layernorm_fwd (kind 0) or rmsnorm_fwd (kind 1, beta and
 * mean ignored) with the kernel forced: SOFTMAX_VARIANT_ROWGROUP (rows of up
 * to 128 chunks of 16 bytes) or SOFTMAX_VARIANT_BLOCK; AUTO chooses. */
int norm_fwd_variant(int kind, const void *x, void *y, int64_t rows, int64_t cols, int dtype, const void *gamma,
                     const void *beta, float eps, float *mean, float *rstd, int variant, softmax_stream_t stream);

/*
 * softmax_query_variant -- the variant softmax_fwd would launch for these
 * arguments on the current device, written to *variant.  Validates the
 * arguments exactly as softmax_fwd does; launches nothing.
 */
int softmax_query_variant(const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
                          int *variant);

/* Device properties the dispatcher reads (one GPU). */
typedef struct {
    int sm_count;           /* multiprocessors */
    int max_smem_optin;     /* max dynamic shared memory per block after opt-in, bytes */
    int cluster_launch;     /* 1 if thread-block cluster launch is supported */
    int l2_bytes;           /* L2 cache size, bytes */
    int cc_major, cc_minor; /* compute capability */
} softmax_device_info;

/* A launch decision: which kernel, and its launch shape. */
typedef struct {
    int variant;            /* softmax_variant chosen (never AUTO) */
    int lanes_per_row;      /* threads that share one row: ROWGROUP G (1..32); BLOCK_TMA
                               32 x warps per row group (32..512); SPLITK_GRID pipelined
                               form: threads of a CTA that fold (the rest write); else 0 */
    int chunks_per_thread;  /* 16-byte chunks each thread caches (ROWGROUP, BLOCK), or loads in
                               flight per thread per streaming step (STREAM, SPLITK); else 0 */
    int rows_per_tile;      /* BLOCK_TMA: consecutive rows moved by one bulk copy; else 0 */
    int stages;             /* BLOCK_TMA: shared-memory tiles in flight per CTA; SPLITK_GRID:
                               ring buffers per CTA (0: streaming form); SPLITK: shared-memory
                               stages per CTA; else 0 */
    int block_threads;      /* threads per CTA */
    int64_t grid_x;         /* CTAs along x */
    int64_t grid_y;         /* CTAs along y (SPLITK: rows; SPLITK_GRID: row groups) */
    int cluster_x;          /* SPLITK: CTAs per cluster (= per row); else 1 */
    int smem_bytes;         /* dynamic shared memory per CTA (BLOCK_TMA, SPLITK_GRID ring form:
                               stages x bytes per stage) */
    int aligned;            /* 1 if every row of x and y starts 16-byte aligned and is a whole
                               number of 16-byte chunks */
    int y_vector;           /* 1 if y rows share x rows' 16-byte phase (vector stores) */
    int back_passes;        /* STREAM: 1 if each pass over a row after the first walks it
                               from the other end, so that a re-read starts on the chunks
                               read last, still in L2 (the dispatcher sets it when the rows
                               in flight hold more than 5/12 of L2; the loads then also
                               carry L2 evict-last / evict-first policies); 0 if every pass
                               walks forward;
                               0 for the other variants.  It changes no 16-bit output bit
                               (fp32: the order of the sum) */
} softmax_launch_plan;

/*
 * softmax_fwd_plan -- launch a caller-supplied plan (for tuning sweeps and
 * benchmarks).  The plan is first checked against the shape, the pointers'
 * alignment and the device: every field must describe a launch that covers
 * each row exactly (e.g. lanes_per_row * chunks_per_thread >= the 16-byte
 * chunks a row spans for ROWGROUP), `aligned` and `y_vector` must match the
 * pointers, and a cluster must fit the device; otherwise
 * SOFTMAX_ERR_INVALID_ARG and nothing is launched.  grid_x may be smaller than
 * the number of rows (or row groups): the kernels loop over rows.
 */
int softmax_fwd_plan(const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                     const softmax_launch_plan *plan, softmax_stream_t stream);

/*
 * softmax_plan -- the dispatcher as a pure host function: the plan that
 * softmax_fwd_variant would launch for these arguments on a device described
 * by *dev.  x and y are only inspected for their addresses (alignment,
 * overlap), never dereferenced, so host addresses may stand in for device
 * ones.  Makes no CUDA call.
 */
int softmax_plan(const softmax_device_info *dev, const void *x, const void *y, int64_t rows,
                 int64_t cols, int dtype, int variant, softmax_launch_plan *plan);

/*
 * softmax_bwd_plan / softmax_masked_plan / norm_plan -- the dispatchers of
 * softmax_bwd_variant, softmax_fwd_masked_variant and norm_fwd_variant as pure
 * host functions, like softmax_plan: the plan those calls would launch for
 * these arguments on a device described by *dev (the mask, scale, causal cut,
 * eps and the mean / rstd outputs do not change the plan and are not taken).
 * Arguments are validated as the launching calls validate them; pointers are
 * only inspected for their addresses.  rows == 0 or cols == 0 gives OK and a
 * zeroed plan.  Makes no CUDA call.
 */
int softmax_bwd_plan(const softmax_device_info *dev, const void *y, const void *dy, const void *dx,
                     int64_t rows, int64_t cols, int dtype, int variant, softmax_launch_plan *plan);
int softmax_masked_plan(const softmax_device_info *dev, const void *x, const void *y, int64_t rows,
                        int64_t cols, int dtype, int variant, softmax_launch_plan *plan);
int norm_plan(const softmax_device_info *dev, int kind, const void *x, const void *y, int64_t rows,
              int64_t cols, int dtype, const void *gamma, const void *beta, int variant,
              softmax_launch_plan *plan);

/* softmax_device_query -- fill *dev for the current CUDA device (cached). */
int softmax_device_query(softmax_device_info *dev);

/*
 * softmax_get_device_error -- read and clear the library's device-side error
 * word on `stream` (the copy is ordered after work already enqueued there and
 * the call synchronises that stream).  *code receives 0 when no kernel
 * reported a problem since the last call, else a nonzero code: the bits of
 * the waits that gave up (1 = bulk-copy arrival, 2 = buffer release, 3 =
 * cluster peer statistics, 4 = a row's grid barrier in SPLITK_GRID).  Kernels
 * that wait bound the wait with %globaltimer; when it runs out they record the
 * code here, drain their own copies in flight and return, so the context
 * stays usable.  A nonzero code also makes this call synchronise the device
 * and clear SPLITK_GRID's barrier scratch.  Returns
 * SOFTMAX_ERR_DEVICE_TIMEOUT if *code is nonzero, SOFTMAX_OK otherwise,
 * SOFTMAX_ERR_CUDA if the copy failed.
 */
int softmax_get_device_error(softmax_stream_t stream, unsigned int *code);

/*
 * softmax_selftest_bounded_wait -- diagnostic for the bounded-wait path above:
 * enqueues on `stream` a one-CTA kernel whose thread waits on a shared-memory
 * mbarrier that nothing arrives on, gives up after limit_us microseconds
 * (1 .. 1000000), records code 1 in the device error word and returns -- no
 * fault, no hang.  A following softmax_get_device_error(stream, &code) then
 * reports SOFTMAX_ERR_DEVICE_TIMEOUT with code 1 and clears the word.
 */
int softmax_selftest_bounded_wait(softmax_stream_t stream, unsigned int limit_us);

/* softmax_last_cuda_error -- the cudaError_t of the last failing CUDA call made
 * by this library on the calling thread (0 if none). */
int softmax_last_cuda_error(void);

/* softmax_strerror -- static description of a softmax_status. */
const char *softmax_strerror(int status);

/* softmax_variant_name -- static name of a softmax_variant ("auto", "rowgroup", ...). */
const char *softmax_variant_name(int variant);

/* softmax_abi_version -- bumped on any incompatible change of this header. */
int softmax_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSD_SOFTMAX_H */
