/*
 * gbce: fused hard-label cross-entropy and row softmax for NVIDIA GB300 (sm_103a).
 *
 * Plain C ABI.  Every pointer argument of the compute calls is DEVICE memory
 * owned by the caller; the library keeps no reference after a call returns.
 * Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream), makes no host synchronisation, and launches only
 * this library's own kernels.  The calling thread's current CUDA device must
 * be the device that owns the buffers.
 *
 * Layout: a matrix argument is M rows of `cols` elements, row r starting at
 * element r * stride of the pointer (row-major, unit column stride, stride in
 * ELEMENTS, cols <= stride <= 2^46; M <= 2^27 - 1; cols < 2^31).  Columns at
 * and beyond `cols` are never read or written.  Row offsets are computed in
 * 64-bit arithmetic.
 *
 * Return value: GBCE_OK (0) or a gbce_status code.  Argument errors are
 * detected on the host before anything is launched and leave every buffer
 * untouched.  Errors that only the device can see (an out-of-range target, a
 * bounded wait that gave up) are raised as sticky per-device flags that
 * gbce_last_error() reports.
 *
 * Bounded waits: the staged kernels wait on mbarriers for their own bulk
 * copies.  Every such wait gives up after 2 s; the CTA then raises
 * GBCE_ERR_TIMEOUT, stops writing results, waits (again within a fixed
 * budget) for the copies it has already issued, and exits, so a failed copy
 * ends the call with an error instead of hanging the device.  Results of a
 * call that raised GBCE_ERR_TIMEOUT are unspecified inside each operand's rows
 * [0, cols) (a row the failing CTA had not finished may be partly written);
 * nothing outside them is written, and the device stays usable.
 */
#ifndef GBCE_H
#define GBCE_H

#include <stdint.h>

#if defined(__GNUC__)
#define GBCE_API __attribute__((visibility("default")))
#else
#define GBCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st *gbce_stream_t;

/* Element types of the logits / softmax operands. */
enum gbce_dtype {
    GBCE_F32 = 0,  /* IEEE binary32 */
    GBCE_BF16 = 1, /* bfloat16; arithmetic is fp32, results are rounded to nearest even */
    GBCE_F16 = 2   /* IEEE binary16; arithmetic is fp32, results rounded to nearest even */
};

/* Bits a call ORs into its own status word (the _ex entry points that take one). */
enum gbce_status_bit {
    GBCE_STATUS_TIMEOUT = 1,  /* one of the call's bounded waits gave up (GBCE_ERR_TIMEOUT) */
    GBCE_STATUS_BAD_TABLE = 2 /* a block-sparse look-up table entry is malformed (GBCE_ERR_BAD_TABLE) */
};

/* Reductions of ce_fwd_bwd_ex (PyTorch CrossEntropyLoss's reduction argument). */
enum gbce_reduction {
    GBCE_MEAN = 0, /* L = sum of row losses / n (n = rows whose target is not ignored) */
    GBCE_SUM = 1,  /* L = sum of row losses */
    GBCE_NONE = 2  /* the row losses themselves, no scalar */
};

enum gbce_status {
    GBCE_OK = 0,
    GBCE_ERR_NULL = 1,        /* a required pointer is NULL */
    GBCE_ERR_SIZE = 2,        /* M < 0, cols < 1, stride < cols, or a size beyond the limits */
    GBCE_ERR_DTYPE = 3,       /* dtype is not a gbce_dtype */
    GBCE_ERR_ALIGN = 4,       /* a pointer is not aligned to its element size */
    GBCE_ERR_CUDA = 5,        /* a CUDA runtime call (allocation, launch) failed */
    GBCE_ERR_BAD_TARGET = 6,  /* device flag: a target outside [0, V) that is not ignore_index */
    GBCE_ERR_TIMEOUT = 7,     /* device flag: a bounded wait on an asynchronous copy gave up */
    GBCE_ERR_NO_DEVICE = 8,   /* no usable CUDA device */
    GBCE_ERR_REDUCTION = 9,   /* reduction is not a gbce_reduction */
    GBCE_ERR_BAD_TABLE = 10   /* device flag: a block-sparse look-up table entry is malformed */
};

/*
 * ce_fwd_bwd -- fused hard-label cross-entropy, forward and backward in one call.
 *
 * Defined by: Liger-Kernel, src/liger_kernel/ops/cross_entropy.py,
 * liger_cross_entropy_kernel (steps 1-6) and LigerCrossEntropyFunction.forward:
 * hard labels, mean reduction over the non-ignored rows, PyTorch
 * CrossEntropyLoss semantics, gradient stored in place over the input.
 *
 *   logits        [M, stride] of dtype, rows of V logits.  READ, then OVERWRITTEN
 *                 IN PLACE with dL/dlogits:
 *                   g[r,i] = (softmax(x_r)_i - [i == t_r]) / n     (t_r != ignore_index)
 *                   g[r,i] = 0                                      (t_r == ignore_index)
 *                 n = number of rows whose target is not ignore_index, over the
 *                 whole call.  Elements outside [0, V) of each row are untouched.
 *   stride        row stride of logits in elements (>= V).
 *   targets       [M] int64 class indices (PyTorch convention), read only.
 *   loss          one float: receives L = sum_r l_r / n with
 *                 l_r = max(x_r) + ln sum_i exp(x_r,i - max(x_r)) - x_r,t_r.
 *                 When n == 0 (M == 0 or every row ignored) L is NaN (0/0).
 *   M, V          rows and classes; M >= 0, 1 <= V < 2^31, M * V may exceed 2^32.
 *   ignore_index  target value that marks a row as ignored (PyTorch uses -100).
 *   dtype         GBCE_F32, GBCE_BF16 or GBCE_F16 (logits; targets are always
 *                 int64).  Arithmetic is fp32 with one rounding per stored value.
 *
 * Accuracy: exp(x - m) is evaluated as exp2((x - m) log2e), the difference
 * formed first, so its error follows the distance |x - m| from the row maximum
 * and not the logits' magnitude; the row loss is (m - x_t) + ln d.  fp32
 * results stay within 1e-5 (relative) of exact for any finite logits (tested
 * with row maxima up to +-1e6 in every kernel regime).
 *
 * A bounded wait that gives up (see above) raises GBCE_ERR_TIMEOUT and makes
 * L NaN; the call's gradient rows are then unspecified as stated above.
 *
 * A target that is neither ignore_index nor in [0, V) leaves its row
 * unmodified, makes L NaN and raises GBCE_ERR_BAD_TARGET in gbce_last_error().
 * Temporary device memory (M floats and a counter) is taken stream-ordered
 * from a library-owned memory pool and returned within the call's stream work.
 * Results are deterministic: the same inputs give the same bits.
 */
GBCE_API int ce_fwd_bwd(void *logits, int64_t stride, const int64_t *targets, float *loss, int64_t M,
               int64_t V, int64_t ignore_index, int dtype, gbce_stream_t stream);

/*
 * ce_fwd_bwd_ex -- ce_fwd_bwd with a reduction, a per-row loss output and the
 * incoming gradient of the loss folded into the in-place gradient.
 *
 * Defined by: Liger-Kernel, src/liger_kernel/ops/cross_entropy.py: the kernel
 * docstring defers to PyTorch's CrossEntropyLoss, whose reduction is 'mean',
 * 'sum' or 'none'; LigerCrossEntropyFunction.backward multiplies the stored
 * gradient by grad_output (element_mul).  Here that multiplication happens in
 * the same pass that writes the gradient, when the caller knows grad_output
 * in advance (e.g. a loss scale).
 *
 *   logits, stride, targets, M, V, ignore_index, dtype: as for ce_fwd_bwd;
 *                 dtype may also be GBCE_F16.  logits is overwritten with
 *                   g[r,i] = (softmax(x_r)_i - [i == t_r]) * k_r,
 *                   k_r = s / n (GBCE_MEAN), s (GBCE_SUM), s_r (GBCE_NONE),
 *                 and 0 for ignored rows.
 *   loss          one float receiving L (GBCE_MEAN: NaN when n == 0; GBCE_SUM: 0
 *                 when M == 0); not used, and may be NULL, for GBCE_NONE.
 *   row_loss      M floats receiving the row losses l_r (0 for ignored rows, NaN
 *                 for an out-of-range target), 16-byte aligned; required for
 *                 GBCE_NONE, optional (NULL) otherwise.  After GBCE_ERR_TIMEOUT
 *                 the row losses of rows the failing CTA had not finished are
 *                 unspecified (a reduced L is NaN).
 *   grad_scale    device floats giving s: NULL means 1; one float for GBCE_MEAN
 *                 and GBCE_SUM; M floats (s_r) for GBCE_NONE.  Read on the device.
 *   reduction     a gbce_reduction, else GBCE_ERR_REDUCTION.
 *
 * ce_fwd_bwd(...) is ce_fwd_bwd_ex(..., loss, NULL, NULL, ..., GBCE_MEAN).
 */
GBCE_API int ce_fwd_bwd_ex(void *logits, int64_t stride, const int64_t *targets, float *loss,
                           float *row_loss, const float *grad_scale, int64_t M, int64_t V,
                           int64_t ignore_index, int dtype, int reduction, gbce_stream_t stream);

/*
 * scale_rows -- x[r, 0:N] *= scale[per_row ? r : 0], in place.
 *
 * Defined by: Liger-Kernel cross_entropy.py, element_mul as applied by
 * LigerCrossEntropyFunction.backward to the gradient stored in place by the
 * forward.  The page skips the call when grad_output == 1 after a host-side
 * comparison (a synchronisation); here the kernel reads the scale on the
 * device and returns at once when a single scale equals 1, so no host sync.
 *
 *   x      [M, stride] of dtype (any gbce_dtype), updated in place.
 *   scale  device floats: one (per_row == 0) or M (per_row != 0).
 */
GBCE_API int scale_rows(void *x, int64_t stride, int64_t M, int64_t N, int dtype,
                        const float *scale, int per_row, gbce_stream_t stream);

/* Largest row count M that ce_fwd_bwd_noalloc accepts. */
#define GBCE_NOALLOC_MAX_ROWS 65536

/*
 * ce_fwd_bwd_noalloc -- ce_fwd_bwd that allocates no device memory.
 *
 * The pages have no counterpart of this entry point.  It is for callers that
 * cannot have a library allocate device memory at call time: processes whose
 * caching allocator has reserved the device's memory up front, serving
 * runtimes that forbid allocation after start-up to keep a fixed memory
 * budget, and devices or drivers without stream-ordered memory pools
 * (cudaDevAttrMemoryPoolsSupported == 0).
 *
 * Arguments, results, layout and errors are those of ce_fwd_bwd, computed by
 * the same kernels.  The temporary storage (the non-ignored count and M row
 * losses) lives instead in one fixed array of static device memory inside
 * this library, about 256 KB, which every GPU that loads the library holds
 * until the process exits.  Hence:
 *   - M > GBCE_NOALLOC_MAX_ROWS is rejected with GBCE_ERR_SIZE before any launch;
 *   - no cudaMalloc, cudaMallocAsync, cudaFree or other allocating call is made;
 *   - every call on a device shares that array and leaves its contents behind;
 *     each call overwrites every entry it reads, so no state carries over, but
 *     calls whose work overlaps on the GPU (on different streams, or from
 *     different host threads) race on it and must be serialised by the caller;
 *   - the first call on each device looks up the array's device address (with
 *     that device current); it may be a call captured into a CUDA graph.
 */
GBCE_API int ce_fwd_bwd_noalloc(void *logits, int64_t stride, const int64_t *targets, float *loss,
                                int64_t M, int64_t V, int64_t ignore_index, int dtype,
                                gbce_stream_t stream);

/*
 * ce_fwd_bwd_host -- ce_fwd_bwd with the logits and targets in host memory
 * and the loss returned to host memory: the end-to-end form of the call.
 *
 *   logits_host [M, host_stride] host memory, read (pinned memory makes the
 *               copies asynchronous; pageable memory works, synchronously).
 *   targets_host [M] int64, host memory, read.
 *   grad        [M, stride] device memory, written: it receives the logits
 *               and then, in place, d(loss)/d(logits) exactly as ce_fwd_bwd
 *               writes them (columns 0..V-1 of each row).
 *   loss_host   one float in host memory: the mean loss, written when the
 *               stream reaches the end of the call (synchronise before reading).
 * The logits are copied in up to 8 row chunks on a library-owned copy stream
 * of the device; each chunk's row kernel waits only for its own chunk, so the
 * copy of chunk k + 1 overlaps the kernel of chunk k.  The copies start after
 * the work already enqueued on `stream`; the call's results are ordered before
 * later work on `stream`.  Scratch (the targets, n, the row losses) comes from
 * the same stream-ordered pool as ce_fwd_bwd.  Argument errors as ce_fwd_bwd,
 * plus GBCE_ERR_SIZE for host_stride < V; device flags through gbce_last_error.
 */
GBCE_API int ce_fwd_bwd_host(const void *logits_host, int64_t host_stride,
                             const int64_t *targets_host, void *grad, int64_t stride,
                             float *loss_host, int64_t M, int64_t V, int64_t ignore_index,
                             int dtype, gbce_stream_t stream);

/*
 * softmax_fwd -- row-wise safe softmax, y = exp(x - max x) / sum exp(x - max x).
 *
 * Defined by: "python sum function examples (triton.language)", _softmax and
 * softmax_kernel (one program per row, separate input and output row strides).
 *
 *   x [M, x_stride] read; y [M, y_stride] written (cols 0..N-1 of each row).
 *   y may be the same buffer as x (same stride): each row is read completely
 *   before any of it is written.  Other partial overlaps are not allowed.
 */
GBCE_API int softmax_fwd(const void *x, int64_t x_stride, void *y, int64_t y_stride, int64_t M, int64_t N,
                int dtype, gbce_stream_t stream);

/*
 * softmax_bwd -- softmax backward, dx = y * (dy - sum(y * dy)) per row.
 *
 * Defined by: "python sum function examples (triton.language)", _backward
 * (fused softmax backward), dense rows and scale 1.
 *
 *   y  [M, y_stride]  softmax output, read.
 *   dy [M, dy_stride] upstream gradient, read.
 *   dx [M, dx_stride] written.  dx may be the same buffer as dy (same stride),
 *   as in the page's in-place store; other overlaps are not allowed.
 */
GBCE_API int softmax_bwd(const void *y, int64_t y_stride, const void *dy, int64_t dy_stride, void *dx,
                int64_t dx_stride, int64_t M, int64_t N, int dtype, gbce_stream_t stream);

/*
 * softmax_fwd_ex, softmax_bwd_ex -- softmax_fwd and softmax_bwd with a status
 * word of the call's own.
 *
 * Defined by: as softmax_fwd and softmax_bwd.  The pages' kernels have no
 * failure path; the status word lets a caller with concurrent calls (several
 * streams or host threads) tell which call failed, where the device flags of
 * gbce_last_error belong to the whole device.
 *
 *   status  NULL (the same as softmax_fwd / softmax_bwd), or one caller-owned
 *           device unsigned int, 4-byte aligned (else GBCE_ERR_ALIGN before any
 *           launch), that the caller clears before the call.  The call ORs
 *           GBCE_STATUS_TIMEOUT into it when one of its bounded waits gave up,
 *           i.e. when it also raises GBCE_ERR_TIMEOUT in the device flags; it
 *           writes nothing else there.  Read it after the call's work on `stream`
 *           has completed.  Other arguments, results and errors: as for
 *           softmax_fwd / softmax_bwd.
 */
GBCE_API int softmax_fwd_ex(const void *x, int64_t x_stride, void *y, int64_t y_stride, int64_t M,
                            int64_t N, int dtype, unsigned int *status, gbce_stream_t stream);
GBCE_API int softmax_bwd_ex(const void *y, int64_t y_stride, const void *dy, int64_t dy_stride,
                            void *dx, int64_t dx_stride, int64_t M, int64_t N, int dtype,
                            unsigned int *status, gbce_stream_t stream);

/*
 * softmax_bwd_bsr -- block-sparse softmax backward through a look-up table,
 * dx = y * (dy - sum(y * dy)) * scale over every row of a block-sparse matrix.
 *
 * Defined by: "python sum function examples (triton.language)", _backward
 * (the block-sparse softmax backward with its look-up table and `scale`).
 *
 * Storage: Z batch items; item z of an operand starts at z * <op>_zstride
 * elements.  Each item holds `nblocks` blocks of block x block elements, block
 * b at b * block^2, row-major inside the block.
 *
 *   lut [lut_len] int32, device memory.  lut[2 rbm] = size and lut[2 rbm + 1] =
 *     offset for block-row rbm = 0 .. n_block_rows-1; the block-row's blocks are
 *     lut[offset + 4 k], k = 0 .. size-1 (entries of 4 ints, block id first;
 *     the other three ints are not read).  Row rxm of block-row rbm (matrix row
 *     rbm * block + rxm) is the concatenation of row rxm of those blocks.  Each
 *     block belongs to one block-row; a block listed twice gives unspecified
 *     values (no memory error).
 *   y  softmax output, read.   dy upstream gradient, read.
 *   dx written at every position the table names, nothing else; dx may be dy
 *     (same zstride), as in the page's in-place store; other overlaps are not
 *     allowed.
 *   block     a power of two, 1 .. 1024.
 *   sizemax   the largest size of any block-row (sizemax * block < 2^31); it
 *             sets the shared-memory plan, so pass the table's true maximum.
 *   scale     multiplies the result.
 * Batch strides are ignored when Z <= 1, else must be >= nblocks * block^2.
 * Argument errors (GBCE_ERR_DTYPE, _SIZE, _NULL, _ALIGN) are returned before
 * any launch.  Z, n_block_rows or sizemax of 0: nothing to do, GBCE_OK.  A
 * block-row whose size is negative or above sizemax, whose entries run past
 * lut_len, or that names a block outside [0, nblocks) is left unwritten for
 * every batch item and raises GBCE_ERR_BAD_TABLE in gbce_last_error();
 * nothing outside the named blocks is read or written.
 */
GBCE_API int softmax_bwd_bsr(const void *y, int64_t y_zstride, const void *dy, int64_t dy_zstride,
                             void *dx, int64_t dx_zstride, const int32_t *lut, int64_t lut_len,
                             int64_t n_block_rows, int64_t nblocks, int64_t block,
                             int64_t sizemax, int64_t Z, float scale, int dtype,
                             gbce_stream_t stream);

/*
 * softmax_bwd_bsr_ex -- softmax_bwd_bsr with a status word of the call's own.
 *
 * Defined by: as softmax_bwd_bsr.  status: NULL (the same as softmax_bwd_bsr),
 * or one caller-owned device unsigned int, 4-byte aligned (else GBCE_ERR_ALIGN
 * before any launch), cleared by the caller; the call ORs GBCE_STATUS_BAD_TABLE
 * into it when it finds a malformed table entry (and raises
 * GBCE_ERR_BAD_TABLE in the device flags), nothing else.  Read it after the
 * call's work on `stream` has completed.
 */
GBCE_API int softmax_bwd_bsr_ex(const void *y, int64_t y_zstride, const void *dy, int64_t dy_zstride,
                                void *dx, int64_t dx_zstride, const int32_t *lut, int64_t lut_len,
                                int64_t n_block_rows, int64_t nblocks, int64_t block,
                                int64_t sizemax, int64_t Z, float scale, int dtype,
                                unsigned int *status, gbce_stream_t stream);

/*
 * gbce_bsr_plan -- the kernel softmax_bwd_bsr uses for `block`, `sizemax` and
 * `dtype` ("bsr_bwd_staged_kernel": one CTA per block-row and batch item, its
 * rows staged in shared memory a slab at a time, *rows_per_slab rows per slab
 * for a block-row of sizemax blocks (shorter block-rows take more);
 * "bsr_bwd_unstaged_kernel": one row per CTA, two passes over global memory,
 * *rows_per_slab = 1; " (element accesses)" appended when `aligned` is 0 or a
 * block row is under 16 bytes).  NULL for invalid arguments.  For tests and
 * diagnostics; no kernel is launched.
 */
GBCE_API const char *gbce_bsr_plan(int64_t block, int64_t sizemax, int dtype, int aligned,
                                   int *rows_per_slab);

/*
 * gbce_plan -- the row-kernel family a call uses for M rows of `cols`
 * elements of `dtype` on the current device: "rows_warp_kernel" (rows of at
 * most 8 KB per operand, one warp per row), "rows_resident_kernel" (at most
 * 64 KB staged per row, one CTA per row), "rows_ring_kernel" (longer rows
 * streamed through a shared-memory ring, *ctas_per_row CTAs of a cluster per
 * row) or "rows_streaming_kernel" (operands whose rows start at different
 * addresses mod 16 bytes: same_phase == 0).  op: 0 ce_fwd_bwd /
 * ce_fwd_bwd_ex, 1 softmax_fwd, 2 softmax_bwd.
 *
 * The plan depends on M only for small batches: when M is at most the
 * device's SM count and rows stage more than 32 KB, the rows take the ring;
 * rows of 64 KB or more per operand are split across the largest cluster (at
 * most 16 CTAs, slices of at least 16 KB) of which M fit on the device at
 * once, so that the whole batch is in flight in one wave.  When no cluster
 * size allows that, the plan is the one for large M.  ce_fwd_bwd_host plans
 * for all of its M rows, like the device call.  Without a usable device the plan for large M is
 * returned.  Returns NULL for invalid arguments (M < 0 included).  For tests
 * and diagnostics; no kernel is launched.
 */
GBCE_API const char *gbce_plan(int op, int64_t M, int64_t cols, int dtype, int same_phase,
                               int *ctas_per_row);

/*
 * gbce_last_error -- synchronise `stream`, then read and clear the current
 * device's sticky error flags.  Returns GBCE_OK, GBCE_ERR_BAD_TARGET,
 * GBCE_ERR_BAD_TABLE or GBCE_ERR_TIMEOUT (the first of these that is set, in
 * this order), or GBCE_ERR_CUDA when the synchronisation itself failed.
 *
 * The flags belong to the DEVICE, not to a stream or a call: every call on
 * the device, from any stream or host thread, raises into the same word, and
 * the read clears it for all of them.  Only `stream` is synchronised, so a
 * flag raised by a call still running on another stream may be reported by a
 * later read instead.  A caller that needs a status per call runs its calls
 * on one stream, or synchronises every stream that used the device and calls
 * this once (the result then covers all of those calls), or uses the _ex
 * entry points, whose status word belongs to the one call (softmax_fwd_ex,
 * softmax_bwd_ex, softmax_bwd_bsr_ex).  The cross-entropy calls also carry
 * their own errors in their result: a bad target or a wait that gave up makes
 * the reduced loss NaN.
 */
GBCE_API int gbce_last_error(gbce_stream_t stream);

/* gbce_status_string -- a static, NUL-terminated description of a status code. */
GBCE_API const char *gbce_status_string(int status);

/*
 * gbce_pool_reserved -- device memory, in bytes, that the library's scratch
 * pool holds on `device` (reserved from the driver and kept for reuse), or 0
 * in *bytes when no call on that device has needed the pool yet.  The pool
 * serves ce_fwd_bwd, ce_fwd_bwd_ex and ce_fwd_bwd_host; ce_fwd_bwd_noalloc
 * and the softmax calls never create it.  For diagnostics; no launch, no sync.
 */
GBCE_API int gbce_pool_reserved(int device, uint64_t *bytes);

/*
 * gbce_test_failure_path -- a test of the bounded waits (no counterpart on the
 * pages).  Makes CTA 0 of every later launch of a staged row kernel
 * (rows_resident_kernel, rows_ring_kernel) on any device leave out its
 * `drop_copy`-th bulk copy (counting from 0; -1 leaves none out, the default).
 * The waits for the missing copy then run out after their 2 s limit and the
 * GBCE_ERR_TIMEOUT path above runs, with no fault and no hang: such a call
 * takes a few seconds.  Takes effect for launches made after it returns.  A
 * process that never calls it never leaves a copy out.
 */
GBCE_API int gbce_test_failure_path(int64_t drop_copy);

/*
 * Kernel timing for benchmarks.  While enabled, every ce_fwd_bwd /
 * softmax_fwd / softmax_bwd call brackets its row kernel (the kernel that
 * streams the logits) with two CUDA events on the call's stream.
 * gbce_timing_read() waits for those events, returns the summed kernel time in
 * milliseconds and the number of bracketed launches, and forgets them.
 * gbce_timing_enable(0) drops unread records.  Not thread safe with
 * concurrent calls from several host threads.
 */
GBCE_API int gbce_timing_enable(int on);
GBCE_API int gbce_timing_read(double *total_ms, int64_t *launches);

#ifdef __cplusplus
}
#endif

#endif /* GBCE_H */
