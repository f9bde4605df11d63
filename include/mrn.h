/*
 * mrn.h -- C ABI of libmrn: RMSNorm, post-norm-then-add and the dual-epsilon
 * sandwich tail on NVIDIA GB300 (sm_103a), hand-written CUDA kernels.
 *
 * Operations (row r of a contiguous row-major [rows x n] matrix, j = 0..n-1):
 *
 *   mrn_rmsnorm             y[r,j]   = x[r,j] * inv(x[r,:]; eps) * gamma[j]
 *   mrn_rmsnorm_then_add    out[r,j] = x[r,j] * inv(x[r,:]; eps) * gamma[j] + residual[r,j]
 *   mrn_norm_residual_norm  out_stream[r,j] = block_out[r,j] * inv(block_out[r,:]; eps_post)
 *                                             * gamma_post[j] + residual[r,j]
 *                           normed[r,j]     = out_stream[r,j] * inv(out_stream[r,:]; eps_pre)
 *                                             * gamma_pre[j]
 *   with inv(v; eps) = 1 / sqrt((1/n) sum_j v_j^2 + eps).
 * Built on the same row reduction (declared further down, same conventions):
 *   mrn_add_rmsnorm, mrn_rmsnorm_then_add_scale, mrn_rmsnorm_q8_1 (Hesper
 *   "RMSNorm Layer" kernels) and the split-norm seam mrn_rmsnorm_seam,
 *   mrn_rmsnorm_unweighted, mrn_seam_scale ("Chapter 12", section 12.7).
 *
 * Sources: "Chapter 12 -- RMSNorm and the dual-epsilon sandwich" section 12.1
 * (definition), 12.2 (two epsilons: 1e-8 for the post norms, 1e-5 for the pre
 * norms), 12.4.3 (the fused tail: hidden += rms_norm(src, eps1) * w1, then
 * output = rms_norm(hidden, eps2) * w2, in one dispatch); the Hesper "RMSNorm
 * Layer" page, rmsNormThenAddKernel / rmsNormThenAddBatchKernel (post norm then
 * residual add, row-major batch) and rmsNormThenAddBatchInPlaceKernel (in-place
 * residual update).
 *
 * Common conventions for the operations
 * -------------------------------------
 * Pointers   All data pointers are CUDA device pointers (or managed memory)
 *            owned by the caller.  The library allocates no memory, keeps no
 *            per-call state and never frees anything.
 * Layout     Row operands are contiguous row-major [rows x n]: element (r, j)
 *            at base + r*n + j.  gamma vectors are [n] and shared by all rows.
 * dtype      MRN_F32: every operand is float.  MRN_BF16: every operand (row
 *            data and gamma) is bfloat16; arithmetic is f32 and each output is
 *            rounded once to bf16 (to nearest, ties to even).  In the bf16
 *            sandwich, normed is computed from the rounded out_stream that is
 *            stored (the split route's publication boundary, section 12.4.4).
 * eps        float, finite and > 0; used as given (the f32 value).
 * Sizes      n >= 1; rows >= 0.  rows == 0 is a no-op that returns MRN_OK
 *            without reading any pointer.  rows * n * element size must fit
 *            in int64.
 * Alignment  Each pointer must be aligned to its element size.  When every
 *            pointer is 16-byte aligned and n * element size is a multiple
 *            of 16, rows are moved in 16-byte vectors.  Otherwise, batches of
 *            the plain, then-add, then-add-scale and sandwich operations whose
 *            row operands and outputs all sit at one offset within 16 bytes
 *            (a row pitch that is not a multiple of 16 bytes on aligned
 *            buffers, or buffers offset alike) are still read as 16-byte
 *            granules: each row's granules are copied whole, including up to
 *            15 bytes before its first and after its last element within the
 *            same granules (never more), and its edge elements are written
 *            one by one.  Everything else moves element-wise.
 * Aliasing   An output may be the very same buffer as a row input (same base
 *            pointer): y == x, out == x or out == residual, out_stream ==
 *            residual (the in-place residual update) or out_stream ==
 *            block_out, normed == block_out or normed == residual.  Any
 *            other overlap -- partial overlaps, two outputs overlapping, an
 *            output overlapping a gamma -- is rejected with MRN_ERR_ALIASING.
 * Stream     Work is enqueued on `stream` (0 = the legacy default stream) and
 *            runs asynchronously; the call returns once it is enqueued.
 * Errors     Argument errors are detected before anything is enqueued; nothing
 *            is written.  MRN_ERR_CUDA means the launch itself failed (see
 *            mrn_last_cuda_error).  Faults during execution surface at the
 *            caller's next synchronisation, as for any CUDA kernel.  Every
 *            wait inside a kernel is bounded (about one second); one that runs
 *            out is counted on the device and reported only by
 *            mrn_wait_timeouts(), never as the status of the call that
 *            enqueued the kernel (that call returned MRN_OK at enqueue time).
 *            The affected rows' outputs are then not written (staged kernels)
 *            or unspecified (cluster reductions of the register kernel).
 * Threads    All entry points are thread-safe.
 */
#ifndef MRN_H
#define MRN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mrn_dtype {
    MRN_F32 = 0,
    MRN_BF16 = 1,
    MRN_F16 = 2    /* IEEE binary16: only as the publication format of the seam
                      operations below; every other use is MRN_ERR_UNSUPPORTED_DTYPE */
} mrn_dtype;

typedef enum mrn_status {
    MRN_OK = 0,
    MRN_ERR_NULL_POINTER = 1,      /* a required pointer is NULL (rows > 0) */
    MRN_ERR_INVALID_SIZE = 2,      /* n < 1, rows < 0, or rows*n*size overflows */
    MRN_ERR_INVALID_EPS = 3,       /* eps not finite or not > 0 */
    MRN_ERR_UNSUPPORTED_DTYPE = 4, /* dtype not MRN_F32 / MRN_BF16 (seam format not
                                      MRN_F16 / MRN_BF16) */
    MRN_ERR_ALIASING = 5,          /* a forbidden overlap between buffers */
    MRN_ERR_MISALIGNED = 6,        /* a pointer not aligned to its element size */
    MRN_ERR_CUDA = 7,              /* the CUDA runtime refused the launch */
    MRN_ERR_INVALID_GEOMETRY = 8   /* a forced geometry cannot cover the row */
    /* A kernel whose bounded wait ran out is never reported as a call status
       (the call has returned long before): only mrn_wait_timeouts() reports it. */
} mrn_status;

/*
 * RMSNorm of every row ("Chapter 12", section 12.1; the ferrite-lineage
 * rms_norm_batch of section 12.4.1 computes the same thing):
 *   x      [rows x n]  input rows
 *   gamma  [n]         per-channel gain
 *   y      [rows x n]  output; may be x itself
 */
mrn_status mrn_rmsnorm(const void *x, const void *gamma, void *y,
                       int64_t rows, int64_t n, float eps,
                       mrn_dtype dtype, cudaStream_t stream);

/*
 * Post norm then residual add (Hesper "RMSNorm Layer", rmsNormThenAddKernel and
 * its row-major batch form rmsNormAddBatchRowsKernel):
 *   x         [rows x n]  the block output that is normalised
 *   gamma     [n]
 *   residual  [rows x n]  added after the norm
 *   out       [rows x n]  may be x or residual itself (in-place residual update,
 *                         rmsNormThenAddBatchInPlaceKernel)
 */
mrn_status mrn_rmsnorm_then_add(const void *x, const void *gamma,
                                const void *residual, void *out,
                                int64_t rows, int64_t n, float eps,
                                mrn_dtype dtype, cudaStream_t stream);

/*
 * Dual-epsilon sandwich tail in one kernel ("Chapter 12", section 12.4.3,
 * muser_fused_norm_residual_rms_norm_32sg; roles: src = block_out,
 * hidden = residual / out_stream, weight1 = gamma_post, weight2 = gamma_pre,
 * eps1 = eps_post (1e-8 on the pages' model), eps2 = eps_pre (1e-5)):
 *   block_out   [rows x n]  sub-block output (attention o_proj or FFN down)
 *   residual    [rows x n]  residual stream before the update
 *   gamma_post  [n]         the post norm's gain
 *   gamma_pre   [n]         the next pre norm's gain
 *   out_stream  [rows x n]  updated stream; may be residual (in place) or block_out
 *   normed      [rows x n]  next sub-block's input; may be block_out or residual,
 *                           never overlapping out_stream
 */
mrn_status mrn_norm_residual_norm(const void *block_out, const void *residual,
                                  const void *gamma_post, const void *gamma_pre,
                                  void *out_stream, void *normed,
                                  int64_t rows, int64_t n,
                                  float eps_post, float eps_pre,
                                  mrn_dtype dtype, cudaStream_t stream);

/*
 * Residual add, then RMSNorm of the sum, in one kernel (Hesper "RMSNorm Layer",
 * residualAddRmsNormKernel / forwardResidualAdd; the pre-norm shape: the stream
 * is updated, then normalised for the next sub-block):
 *   residual_out[r,j] = a[r,j] + b[r,j]
 *   normed[r,j]       = residual_out[r,j] * inv(residual_out[r,:]; eps) * gamma[j]
 *   a, b          [rows x n]  the two summands (stream and sub-block output)
 *   gamma         [n]
 *   residual_out  [rows x n]  the sum; may be a or b (in-place accumulate)
 *   normed        [rows x n]  may be a or b, never overlapping residual_out
 * bf16: the sum is rounded once to bf16, stored, and that rounded value is
 * normalised (the same publication boundary as the sandwich's stream).
 */
mrn_status mrn_add_rmsnorm(const void *a, const void *b, const void *gamma,
                           void *residual_out, void *normed,
                           int64_t rows, int64_t n, float eps,
                           mrn_dtype dtype, cudaStream_t stream);

/*
 * Post norm, residual add, then a broadcast scalar (Hesper "RMSNorm Layer",
 * rmsNormThenAddThenBroadcastScaleKernel; a per-layer output scale):
 *   out[r,j] = (x[r,j] * inv(x[r,:]; eps) * gamma[j] + residual[r,j]) * out_scale[0]
 *   out_scale  one element of `dtype` in device memory, read by the kernel
 *   out        [rows x n]  may be x or residual; must not overlap out_scale
 * Arithmetic: fma(x * inv, gamma, residual) in f32, times out_scale, rounded
 * once to the output type.
 */
mrn_status mrn_rmsnorm_then_add_scale(const void *x, const void *gamma, const void *residual,
                                      const void *out_scale, void *out,
                                      int64_t rows, int64_t n, float eps,
                                      mrn_dtype dtype, cudaStream_t stream);

/*
 * RMSNorm fused with Q8_1 block quantisation (Hesper "RMSNorm Layer",
 * fusedRMSNormQ8_1Kernel: the norm's output goes straight to the quantised
 * input of the next matvec, with no f32 round trip through memory):
 *   x_normed[j] = x[r,j] * gamma[j] * inv(x[r,:]; eps)            (f32)
 *   per block of 32 consecutive elements of a row:
 *     d = max |x_normed| / 127,  q = round(x_normed / d)  (nearest, ties to
 *     even; clamped to [-128, 127]; q = 0 and d = 0 for an all-zero block)
 *   x       [rows x n]  f32 or bf16 (dtype); n must be a multiple of 32
 *   gamma   [n]         same dtype
 *   blocks  [rows x n/32] blocks of 36 bytes: f16 d (bytes 0-1), f16 s = 0
 *           (bytes 2-3; unused by the page's consumer), int8 q[32]
 *           (bytes 4-35); 4-byte aligned; must not overlap x or gamma
 * n % 32 != 0 gives MRN_ERR_INVALID_SIZE.
 */
mrn_status mrn_rmsnorm_q8_1(const void *x, const void *gamma, void *blocks,
                            int64_t rows, int64_t n, float eps,
                            mrn_dtype dtype, cudaStream_t stream);

/*
 * Split-norm seam: the rounding point between the weightless norm and the
 * weight multiply kept ("Chapter 12", section 12.7, the cross-vendor seam: a
 * producer that publishes the unweighted norm in F16 and applies its scale as
 * a second F16 operation; a receiver that fuses the two loses that rounding
 * point).  S is the 16-bit publication format `seam` (MRN_F16 or MRN_BF16),
 * S(v) rounds an f32 value to S (nearest, ties to even; overflow gives
 * infinity, gradual underflow).
 *   mrn_rmsnorm_unweighted  u[r,j] = S(x[r,j] * inv(x[r,:]; eps))
 *   mrn_seam_scale          y[r,j] = S(u[r,j] * gamma[j])
 *   mrn_rmsnorm_seam        y[r,j] = S(S(x[r,j] * inv(x[r,:]; eps)) * gamma[j])
 * The weight multiply is the IEEE multiply of S (the exact product of two S
 * values rounded once).  The fused form gives, bit for bit, what the two split
 * operations give on the same rows: the reduction (hence inv) is the same for
 * the fused and the weightless call.
 *   x      [rows x n]  f32 or bf16 (dtype)
 *   gamma  [n]         16-bit values of S
 *   u, y   [rows x n]  16-bit values of S; y may be x itself when dtype is
 *                      MRN_BF16 (same element positions), and mrn_seam_scale's
 *                      y may be u itself; no other overlap is allowed
 * Vector paths need 16-byte aligned pointers and n * element size (of x; of
 * u for mrn_seam_scale) a multiple of 16; otherwise element-wise.
 */
mrn_status mrn_rmsnorm_seam(const void *x, const void *gamma, void *y,
                            int64_t rows, int64_t n, float eps,
                            mrn_dtype dtype, mrn_dtype seam, cudaStream_t stream);
mrn_status mrn_rmsnorm_unweighted(const void *x, void *u, int64_t rows, int64_t n, float eps,
                                  mrn_dtype dtype, mrn_dtype seam, cudaStream_t stream);
mrn_status mrn_seam_scale(const void *u, const void *gamma, void *y, int64_t rows, int64_t n,
                          mrn_dtype seam, cudaStream_t stream);

/* Static, human-readable name of a status code; never NULL. */
const char *mrn_status_string(mrn_status status);

/* cudaError_t of the most recent MRN_ERR_CUDA returned on the calling thread
 * (0 if none). */
int mrn_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Introspection and test hooks.  These are not on the pages: they expose the
 * kernel geometry the library picks so that tests can drive every variant
 * and benchmarks can report it.                                              */

typedef enum mrn_op {
    MRN_OP_RMSNORM = 0,
    MRN_OP_THEN_ADD = 1,
    MRN_OP_SANDWICH = 2,
    MRN_OP_ADD_RMSNORM = 3,
    MRN_OP_THEN_ADD_SCALE = 4,
    MRN_OP_RMSNORM_Q8_1 = 5,
    MRN_OP_RMSNORM_SEAM = 6,       /* mrn_rmsnorm_seam (either format) */
    MRN_OP_RMSNORM_UNWEIGHTED = 7  /* mrn_rmsnorm_unweighted (either format) */
} mrn_op;

typedef enum mrn_geometry_kind {
    MRN_GEOM_AUTO = 0,          /* (for mrn_force_geometry) let the library choose */
    MRN_GEOM_ROWS_PER_WARP = 1, /* lanes_per_row (1..32) lanes per row, several rows
                                   per CTA of `threads` (a multiple of 32 up to 256;
                                   0 when forced: 256), shuffle-only reduction */
    MRN_GEOM_CTA = 2,           /* one row per CTA, or per thread-block cluster of
                                   `cluster` CTAs whose partial sums travel as
                                   st.async messages to the peers' shared memory;
                                   row held in registers */
    MRN_GEOM_STREAM = 3,        /* one row per CTA, or per cluster of `cluster` CTAs
                                   each looping over its slice of the row: any n */
    MRN_GEOM_TMA = 4,           /* persistent CTAs; `stages` future rows are copied
                                   into shared memory by cp.async.bulk while the
                                   current one is reduced; gammas kept in shared
                                   memory; needs 16-byte aligned rows.  cluster > 1
                                   (groups 1; plain, then-add, then-add-scale and
                                   the sandwich): a cluster per row, each CTA
                                   staging a 16-byte-multiple slice, the partial
                                   sums exchanged as st.async messages */
    MRN_GEOM_Q8_BLOCKS = 5      /* RMSNorm + Q8_1 only: one row per CTA, `k` (1 or 2)
                                   whole 32-element blocks per thread, `threads` <= 512;
                                   needs 16-byte aligned rows */
} mrn_geometry_kind;

typedef struct mrn_geometry {
    int32_t kind;          /* mrn_geometry_kind */
    int32_t vec;           /* elements per load: 16 / element size, or 1 */
    int32_t k;             /* loads per operand per thread (register slots) */
    int32_t threads;       /* threads per CTA */
    int32_t cluster;       /* CTAs per row, 1..16 (MRN_GEOM_CTA, MRN_GEOM_TMA or
                              MRN_GEOM_STREAM) */
    int32_t lanes_per_row; /* threads per row for MRN_GEOM_ROWS_PER_WARP */
    int32_t rows_per_cta;  /* rows one CTA handles at a time */
    int32_t stages;        /* MRN_GEOM_TMA: rows staged in shared memory (1..8) */
    int32_t ctas;          /* MRN_GEOM_TMA: persistent CTAs (0 = fill the device) */
    int32_t groups;        /* MRN_GEOM_TMA: warp groups per CTA (1 or 2), each
                              reducing its own rows; threads is the CTA total */
    int32_t edge;          /* MRN_GEOM_TMA, cluster 1, groups 2: rows that are not
                              16-byte aligned (plain, then-add, then-add-scale,
                              sandwich; every row operand and output at one offset
                              within 16 bytes), each staged as the 16-byte granules
                              that cover it, the edge elements masked and stored one
                              by one; k * threads / 2 must cover
                              (n * size + 15) / 16 + 1 granules */
} mrn_geometry;

/*
 * The geometry an operation would launch with.  aligned16: 1 states that all
 * pointers would be 16-byte aligned; 2 that they would not, but that every
 * row operand and output would sit at one offset within 16 bytes; 0 neither.
 * sm_count 0 means: ask the current device; a positive value is used as
 * given (lets host-only tests query).  The thread's forced geometry, if any,
 * is reported instead.
 */
mrn_status mrn_query_geometry(mrn_op op, int64_t rows, int64_t n, mrn_dtype dtype,
                              int32_t aligned16, int32_t sm_count, mrn_geometry *out);

/*
 * Force the geometry of the calling thread's later calls (NULL or kind
 * MRN_GEOM_AUTO restores the automatic choice).  Fields 0 mean "automatic"
 * for vec.  A forced geometry that cannot cover a call's row makes that call
 * return MRN_ERR_INVALID_GEOMETRY.  The geometry is checked for internal
 * consistency here (MRN_ERR_INVALID_GEOMETRY if not).
 */
mrn_status mrn_force_geometry(const mrn_geometry *geometry);

/* Number of kernels this library has launched in the process (all threads). */
uint64_t mrn_launch_count(void);

/*
 * Launch options of the calling thread's later calls (default MRN_LAUNCH_PDL;
 * 0 = plain stream-ordered launches).
 *   MRN_LAUNCH_PDL  programmatic dependent launch: a kernel may be scheduled
 *                   before the previous kernel on the stream has finished.
 *                   Every kernel of this library first waits for that
 *                   previous grid to complete and publish its memory
 *                   (griddepcontrol.wait), so results are unchanged; the
 *                   launch latency of a call overlaps the previous kernel
 *                   instead of following it (measured on GB300: ~2 us per
 *                   call in a chain of 4096 x 6656 sandwich calls, ~0.2 us
 *                   per decode call in a CUDA graph).  The previous kernel
 *                   need not be ours; a kernel launched after ours without
 *                   the attribute is ordered as usual.
 *   MRN_LAUNCH_TEST_WAIT_TIMEOUT
 *                   test hook, never for use: the first wait of every CTA
 *                   of the staged kernels (MRN_GEOM_TMA, staged
 *                   MRN_GEOM_Q8_BLOCKS: its gamma copy) and of cluster
 *                   reductions in MRN_GEOM_CTA (its first message exchange)
 *                   expects 16 bytes more than ever arrive, so it runs out
 *                   after about one second.  The staged kernels then write
 *                   nothing; the register kernel's outputs are unspecified.
 *                   mrn_wait_timeouts() reports the waits; the context stays
 *                   usable.  Lets a test drive the timeout path with no fault.
 * Unknown bits give MRN_ERR_INVALID_GEOMETRY.  Not on the pages: a launch
 * option of this library.
 */
#define MRN_LAUNCH_PDL 1u
#define MRN_LAUNCH_TEST_WAIT_TIMEOUT 0x80000000u
mrn_status mrn_set_launch_options(uint32_t options);
uint32_t mrn_launch_options(void);

/*
 * Number of bounded waits (on the shared-memory copy barriers of the staged
 * kernels and the message barriers of cluster reductions) that ran out on the
 * current device since the previous mrn_wait_timeouts() call on that device;
 * -1 if the count could not be read.  This is the only place a timeout is
 * reported: no entry point returns a status for it.  The device-side counts
 * only grow; the library keeps the last value it reported per device (under
 * a lock), so a timeout counted while this function runs is reported by the
 * next call, never lost.  Every wait gives up after about one second of wall
 * time (%globaltimer, which also runs while the context is time-sliced out on
 * a shared GPU); a staged CTA then drains its copies and returns without
 * writing its remaining rows, so the context stays usable.
 * Synchronises the device (it reads device memory with cudaMemcpyFromSymbol).
 * Not on the pages: a diagnostic of this library.
 */
int mrn_wait_timeouts(void);

#ifdef __cplusplus
}
#endif

#endif /* MRN_H */
