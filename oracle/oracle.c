/*
 * Double-precision CPU oracle for the fused hard-label cross-entropy and the
 * row-wise softmax forward/backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Every function is the plain textbook definition, written out row by row in
 * double precision, with no blocking, fusion or online recurrence:
 *
 *   m   = max_i x_i
 *   Z   = sum_i exp(x_i - m)                (compensated sum, index order)
 *   p_i = exp(x_i - m) / Z
 *   l_r = m + ln Z - x_y                    (= -ln p_y)
 *   g_i = (p_i - [i == y]) / n              (n = number of non-ignored rows)
 *   L   = (sum over non-ignored rows of l_r) / n
 *
 * Sources, by page and section:
 *   - Liger-Kernel, src/liger_kernel/ops/cross_entropy.py,
 *     liger_cross_entropy_kernel docstring: hard labels with mean reduction,
 *     following PyTorch's CrossEntropyLoss.
 *   - same kernel, steps 1-2: a row whose target equals ignore_index gets an
 *     all-zero gradient and contributes no loss.
 *   - same kernel, step 4 comment: dx_i = softmax(x_i)/N for i != y and
 *     dx_y = (softmax(x_y) - 1)/N, N = number of non-ignored rows in the batch.
 *   - same kernel, step 5 comment: loss = -(x_y - max(x) - log sum e^(x-max)).
 *   - LigerCrossEntropyFunction.forward: n_non_ignore counts targets that
 *     differ from ignore_index over the whole batch; the loss is the sum of the
 *     per-row losses divided by it.
 *   - "python sum function examples (triton.language)", _softmax and
 *     softmax_kernel: y = exp(x - max x) / sum exp(x - max x) per row.
 *   - same page, _backward (block-sparse softmax backward), dense math with
 *     scale 1: dx = y * (dy - sum(y * dy)).
 *   - same page, _backward with its look-up table: the rows of a block-sparse
 *     matrix are gathered through the table and the result is multiplied by
 *     `scale`; see oracle_softmax_bwd_bsr below.
 *   - Liger-Kernel, LigerCrossEntropyFunction.backward and element_mul: the
 *     stored gradient is multiplied by the incoming grad_output when that is
 *     not 1.
 *   - PyTorch's CrossEntropyLoss, which the kernel docstring defers to, also
 *     defines reduction = 'sum' (L = sum of the row losses, gradient rows not
 *     divided by n) and 'none' (the row losses themselves; the gradient of
 *     sum_r w_r l_r for per-row weights w_r).
 *
 * Readings where the pages are silent:
 *   - n == 0 (every row ignored): the mean is 0/0 = NaN and every gradient row
 *     is zero, as each row takes the ignore exit.
 *   - a target outside [0, V) that is not ignore_index: the row's loss is NaN,
 *     its gradient row is the unmodified input, and the row is counted as bad.
 *     Such a row still counts toward n (n counts targets != ignore_index).
 *   - bf16 and fp16 inputs are widened exactly to double before any arithmetic.
 *   - the gradient of a call is (p - onehot) * k_r with k_r = s / n (mean),
 *     s (sum) or s_r (none), where s (or s_r) is the incoming grad_output
 *     (1 when none is given).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };
enum { ORACLE_MEAN = 0, ORACLE_SUM = 1, ORACLE_NONE = 2 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 * exponent 0 holds zero and the subnormals (fraction * 2^-24), exponent 31
 * holds infinities (fraction 0) and NaNs. */
static double half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int exp = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (exp == 0)
        v = ldexp((double)frac, -24);
    else if (exp == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 1024), exp - 25);
    return sign ? -v : v;
}

/* Read element idx of a row stored as fp32 or as raw bf16 bits, widened
 * exactly to double. */
static double load_elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    if (dtype == ORACLE_F16)
        return half_to_double(((const uint16_t *)base)[idx]);
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Neumaier's compensated summation (Neumaier 1974), summed in index order. */
typedef struct {
    double s, c;
} csum_t;

/* Exposed for the tests: the exact widening of n stored values to double. */
int oracle_widen(const void *src, int dtype, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = load_elem(src, dtype, i);
    return 0;
}

static void csum_add(csum_t *a, double v)
{
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v))
        a->c += (a->s - t) + v;
    else
        a->c += (v - t) + a->s;
    a->s = t;
}

static double csum_value(const csum_t *a) { return a->s + a->c; }

int oracle_ce_count(const int64_t *targets, int64_t M, int64_t V, int64_t ignore_index,
                    int64_t *n_out, int64_t *bad_out)
{
    int64_t n = 0, bad = 0;
    for (int64_t r = 0; r < M; ++r) {
        int64_t y = targets[r];
        if (y == ignore_index)
            continue;
        ++n;
        if (y < 0 || y >= V)
            ++bad;
    }
    if (n_out)
        *n_out = n;
    if (bad_out)
        *bad_out = bad;
    return 0;
}

/* One cross-entropy row.  x: the row's first element; grad: V doubles or NULL;
 * k: the factor of this row's gradient ((p - onehot) * k). */
static void ce_row(const void *x, int dtype, int64_t V, int64_t y, int64_t ignore_index,
                   double k, double *grad, double *loss)
{
    if (y == ignore_index) {
        if (grad)
            for (int64_t i = 0; i < V; ++i)
                grad[i] = 0.0;
        *loss = 0.0;
        return;
    }
    if (y < 0 || y >= V) {
        if (grad)
            for (int64_t i = 0; i < V; ++i)
                grad[i] = load_elem(x, dtype, i);
        *loss = NAN;
        return;
    }
    /* pass 1: the maximum */
    double m = -INFINITY;
    for (int64_t i = 0; i < V; ++i) {
        double v = load_elem(x, dtype, i);
        if (v > m)
            m = v;
    }
    /* pass 2: the normaliser */
    csum_t z = {0.0, 0.0};
    for (int64_t i = 0; i < V; ++i)
        csum_add(&z, exp(load_elem(x, dtype, i) - m));
    double Z = csum_value(&z);
    /* the row loss, -ln p_y */
    *loss = m + log(Z) - load_elem(x, dtype, y);
    /* pass 3: the gradient */
    if (grad) {
        for (int64_t i = 0; i < V; ++i) {
            double p = exp(load_elem(x, dtype, i) - m) / Z;
            double onehot = (i == y) ? 1.0 : 0.0;
            grad[i] = (p - onehot) * k;
        }
    }
}

static void softmax_fwd_row(const void *x, int dtype, int64_t N, double *y)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < N; ++i) {
        double v = load_elem(x, dtype, i);
        if (v > m)
            m = v;
    }
    csum_t z = {0.0, 0.0};
    for (int64_t i = 0; i < N; ++i)
        csum_add(&z, exp(load_elem(x, dtype, i) - m));
    double Z = csum_value(&z);
    for (int64_t i = 0; i < N; ++i)
        y[i] = exp(load_elem(x, dtype, i) - m) / Z;
}

static void softmax_bwd_row(const void *y, const void *dy, int dtype, int64_t N, double *dx)
{
    csum_t s = {0.0, 0.0};
    for (int64_t i = 0; i < N; ++i)
        csum_add(&s, load_elem(y, dtype, i) * load_elem(dy, dtype, i));
    double S = csum_value(&s);
    for (int64_t i = 0; i < N; ++i)
        dx[i] = load_elem(y, dtype, i) * (load_elem(dy, dtype, i) - S);
}

/* ---- a plain parallel-for over the requested rows (rows are independent) ---- */

enum { JOB_CE = 0, JOB_SM_FWD = 1, JOB_SM_BWD = 2 };

typedef struct {
    int kind, dtype;
    const void *a;     /* logits, x, or y */
    int64_t a_stride;
    const void *b;     /* dy for the softmax backward */
    int64_t b_stride;
    const int64_t *targets;
    int64_t ncols, ignore_index, n;
    int reduction;
    const double *grad_scale; /* NULL: 1; else one value, or one per row (none) */
    const int64_t *rows; /* NULL: rows 0..nrows-1 */
    int64_t nrows;
    double *out;       /* nrows x ncols, or NULL (cross-entropy only) */
    double *row_loss;  /* nrows (cross-entropy only) */
    int64_t begin, end;
} job_t;

static size_t elem_size(int dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

static int valid_dtype(int dtype)
{
    return dtype == ORACLE_F32 || dtype == ORACLE_BF16 || dtype == ORACLE_F16;
}

static void *run_job(void *arg)
{
    job_t *j = (job_t *)arg;
    size_t es = elem_size(j->dtype);
    for (int64_t k = j->begin; k < j->end; ++k) {
        int64_t r = j->rows ? j->rows[k] : k;
        const char *ra = (const char *)j->a + (size_t)r * (size_t)j->a_stride * es;
        double *o = j->out ? j->out + (size_t)k * (size_t)j->ncols : NULL;
        if (j->kind == JOB_CE) {
            double s = 1.0;
            if (j->grad_scale)
                s = j->reduction == ORACLE_NONE ? j->grad_scale[r] : j->grad_scale[0];
            const double kf = j->reduction == ORACLE_MEAN ? s / (double)j->n : s;
            ce_row(ra, j->dtype, j->ncols, j->targets[r], j->ignore_index, kf, o,
                   &j->row_loss[k]);
        } else if (j->kind == JOB_SM_FWD) {
            softmax_fwd_row(ra, j->dtype, j->ncols, o);
        } else {
            const char *rb = (const char *)j->b + (size_t)r * (size_t)j->b_stride * es;
            softmax_bwd_row(ra, rb, j->dtype, j->ncols, o);
        }
    }
    return NULL;
}

static int run_parallel(const job_t *proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > proto->nrows)
        nthreads = proto->nrows > 0 ? (int)proto->nrows : 1;
    job_t jobs[256];
    pthread_t tids[256];
    int64_t per = (proto->nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].begin = (int64_t)t * per;
        jobs[t].end = jobs[t].begin + per < proto->nrows ? jobs[t].begin + per : proto->nrows;
        if (jobs[t].begin > jobs[t].end)
            jobs[t].begin = jobs[t].end;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_job, &jobs[t]) != 0) {
            /* run the remaining ranges on this thread instead */
            for (int u = t; u < nthreads; ++u)
                run_job(&jobs[u]);
            break;
        }
        started = t;
    }
    run_job(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    return 0;
}

/* Cross-entropy rows.  rows[k] (or k when rows is NULL) names the input row;
 * grad (nrows x V doubles, or NULL) and row_loss (nrows doubles) are indexed by
 * k.  n is the batch-wide non-ignored count from oracle_ce_count; reduction
 * and grad_scale (NULL, one value, or M values for ORACLE_NONE, indexed by the
 * input row) set the gradient factor. */
int oracle_ce_rows_ex(const void *logits, int dtype, int64_t stride, const int64_t *targets,
                      int64_t V, int64_t ignore_index, int64_t n, int reduction,
                      const double *grad_scale, const int64_t *rows, int64_t nrows, double *grad,
                      double *row_loss, int nthreads)
{
    if (reduction != ORACLE_MEAN && reduction != ORACLE_SUM && reduction != ORACLE_NONE)
        return 1;
    if (!logits || !targets || !row_loss || V < 1 || stride < V || nrows < 0)
        return 1;
    if (!valid_dtype(dtype))
        return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.kind = JOB_CE;
    j.dtype = dtype;
    j.a = logits;
    j.a_stride = stride;
    j.targets = targets;
    j.ncols = V;
    j.ignore_index = ignore_index;
    j.n = n;
    j.reduction = reduction;
    j.grad_scale = grad_scale;
    j.rows = rows;
    j.nrows = nrows;
    j.out = grad;
    j.row_loss = row_loss;
    return run_parallel(&j, nthreads);
}

/* The mean-reduced call without a grad_output (the fused forward+backward). */
int oracle_ce_rows(const void *logits, int dtype, int64_t stride, const int64_t *targets,
                   int64_t V, int64_t ignore_index, int64_t n, const int64_t *rows,
                   int64_t nrows, double *grad, double *row_loss, int nthreads)
{
    return oracle_ce_rows_ex(logits, dtype, stride, targets, V, ignore_index, n, ORACLE_MEAN, NULL,
                             rows, nrows, grad, row_loss, nthreads);
}

/* L = sum_r row_loss[r] / n over all M rows (ignored rows hold 0). */
double oracle_ce_mean(const double *row_loss, int64_t M, int64_t n)
{
    csum_t s = {0.0, 0.0};
    for (int64_t r = 0; r < M; ++r)
        csum_add(&s, row_loss[r]);
    return csum_value(&s) / (double)n;
}

/* L = sum_r row_loss[r] over all M rows (reduction = 'sum'). */
double oracle_ce_sum(const double *row_loss, int64_t M)
{
    csum_t s = {0.0, 0.0};
    for (int64_t r = 0; r < M; ++r)
        csum_add(&s, row_loss[r]);
    return csum_value(&s);
}

int oracle_softmax_fwd_rows(const void *x, int dtype, int64_t stride, int64_t N,
                            const int64_t *rows, int64_t nrows, double *y, int nthreads)
{
    if (!x || !y || N < 1 || stride < N || nrows < 0)
        return 1;
    if (!valid_dtype(dtype))
        return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.kind = JOB_SM_FWD;
    j.dtype = dtype;
    j.a = x;
    j.a_stride = stride;
    j.ncols = N;
    j.rows = rows;
    j.nrows = nrows;
    j.out = y;
    return run_parallel(&j, nthreads);
}

int oracle_softmax_bwd_rows(const void *y, int64_t y_stride, const void *dy, int64_t dy_stride,
                            int dtype, int64_t N, const int64_t *rows, int64_t nrows, double *dx,
                            int nthreads)
{
    if (!y || !dy || !dx || N < 1 || y_stride < N || dy_stride < N || nrows < 0)
        return 1;
    if (!valid_dtype(dtype))
        return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.kind = JOB_SM_BWD;
    j.dtype = dtype;
    j.a = y;
    j.a_stride = y_stride;
    j.b = dy;
    j.b_stride = dy_stride;
    j.ncols = N;
    j.rows = rows;
    j.nrows = nrows;
    j.out = dx;
    return run_parallel(&j, nthreads);
}

/* Block-sparse softmax backward ("python sum function examples
 * (triton.language)", _backward): the softmax output y and the upstream
 * gradient dy of a block-sparse matrix, stored block by block.
 *
 * Storage: batch item z starts at z * zstride elements; block b of it holds a
 * block x block tile, row-major, at b * block^2.  The table `lut` (int32)
 * starts with one (size, offset) pair per block-row rbm; the row's blocks are
 * lut[offset + 4 * rbn] for rbn = 0 .. size-1 (the other three ints of each
 * entry are not read here).  Row pidhm = rbm * block + rxm of the matrix is
 * the concatenation, over rbn, of row rxm of those blocks.  For each batch
 * item and each row:
 *
 *   s    = sum over the row's elements of y * dy
 *   dx_i = y_i * (dy_i - s) * scale
 *
 * dx (Z x zstride doubles, filled by the caller) receives the results at the
 * positions the table names; other positions are left as they are.
 *
 * Readings where the page is silent: a block-row whose size is negative or
 * above sizemax, whose entries run outside the table, or that names a block
 * outside [0, nblocks) is bad: none of its rows is written, for any batch
 * item, and it is counted in *bad.  A size of 0 writes nothing.
 * block_rows (NULL: all n_block_rows) lists the block-rows to compute. */
/* Element rxn of row rxm of block `blockid`: blocks are block x block tiles,
 * row-major, one after another. */
static int64_t bsr_index(int64_t blockid, int64_t rxm, int64_t rxn, int64_t block)
{
    return blockid * block * block + rxm * block + rxn;
}

/* The block id of entry rbn of a block-row whose entries start at `offset`:
 * each entry is 4 ints, the block id first. */
static int64_t bsr_block_id(const int32_t *lut, int64_t offset, int64_t rbn)
{
    return lut[offset + 4 * rbn];
}

int oracle_softmax_bwd_bsr(const void *y, int64_t y_zstride, const void *dy, int64_t dy_zstride,
                           int dtype, const int32_t *lut, int64_t lut_len, int64_t n_block_rows,
                           int64_t nblocks, int64_t block, int64_t sizemax, int64_t Z,
                           double scale, const int64_t *block_rows, int64_t n_listed,
                           double *dx, int64_t dx_zstride, int64_t *bad)
{
    if (!y || !dy || !dx || !lut || !bad || block < 1 || Z < 0 || n_block_rows < 0 ||
        nblocks < 0 || sizemax < 0 || lut_len < 2 * n_block_rows || !valid_dtype(dtype))
        return 1;
    const int64_t bb = block * block;
    if ((Z > 1 && (y_zstride < nblocks * bb || dy_zstride < nblocks * bb ||
                   dx_zstride < nblocks * bb)))
        return 1;
    const int64_t count = block_rows ? n_listed : n_block_rows;
    *bad = 0;
    for (int64_t q = 0; q < count; ++q) {
        const int64_t rbm = block_rows ? block_rows[q] : q;
        if (rbm < 0 || rbm >= n_block_rows)
            return 1;
        const int64_t size = lut[2 * rbm];
        const int64_t offset = lut[2 * rbm + 1];
        int ok = size >= 0 && size <= sizemax;
        if (ok && size > 0)
            ok = offset >= 0 && offset + 4 * (size - 1) < lut_len;
        for (int64_t rbn = 0; ok && rbn < size; ++rbn) {
            const int64_t blockid = bsr_block_id(lut, offset, rbn);
            ok = blockid >= 0 && blockid < nblocks;
        }
        if (!ok) {
            ++*bad;
            continue;
        }
        for (int64_t z = 0; z < Z; ++z) {
            for (int64_t rxm = 0; rxm < block; ++rxm) {
                /* s = sum of y * dy over the row's stored elements */
                csum_t s = {0.0, 0.0};
                for (int64_t rbn = 0; rbn < size; ++rbn) {
                    const int64_t blockid = bsr_block_id(lut, offset, rbn);
                    for (int64_t rxn = 0; rxn < block; ++rxn) {
                        const int64_t e = bsr_index(blockid, rxm, rxn, block);
                        csum_add(&s, load_elem(y, dtype, z * y_zstride + e) *
                                         load_elem(dy, dtype, z * dy_zstride + e));
                    }
                }
                const double S = csum_value(&s);
                /* dx = y * (dy - s) * scale over the same elements */
                for (int64_t rbn = 0; rbn < size; ++rbn) {
                    const int64_t blockid = bsr_block_id(lut, offset, rbn);
                    for (int64_t rxn = 0; rxn < block; ++rxn) {
                        const int64_t e = bsr_index(blockid, rxm, rxn, block);
                        dx[z * dx_zstride + e] = load_elem(y, dtype, z * y_zstride + e) *
                                                 (load_elem(dy, dtype, z * dy_zstride + e) - S) *
                                                 scale;
                    }
                }
            }
        }
    }
    return 0;
}
