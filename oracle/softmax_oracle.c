/*
 * softmax_oracle.c -- the fp64 CPU oracle for row-wise safe softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * tests/, __graft_entry__.smoke() and the cpu_baseline / reference legs of
 * bench.py may load it.  It shares no code, header, table or constant with the
 * CUDA library under online_softmax_dispatcher_gb300/csrc, and neither side
 * includes or links the other.  The only agreement between the two is the
 * numeric dtype code (0 = fp32, 1 = fp16, 2 = bf16), which is an interface.
 *
 * What it computes (plain definitions, written out; no blocking, fusion or
 * reordering beyond what the definitions state):
 *
 *   safe softmax along the last dimension of a row-major [rows, cols] array,
 *       m   = max_j x_j
 *       s   = sum_j exp(x_j - m)
 *       y_j = exp(x_j - m) / s
 *   as stated in
 *     - "[CUDA] safe online softmax" (wingedge777.com), section 1 "safe online
 *       softmax", the safe_softmax listing (max, then exp(x - max), then divide
 *       by the sum);
 *     - the HIP softmax tutorial (forum.sourcefind.cn), section 1 "Softmax
 *       operator definition", the numerically stable formula
 *       y_i = e^(x_i - max(x)) / sum_j e^(x_j - max(x));
 *     - "Softmax on DCU: from 2.34 ms to 0.62 ms" (czchanglian.com), section 1,
 *       which motivates the max subtraction (exp overflows without it).
 *   All arithmetic is IEEE binary64 in the C default rounding mode
 *   (round-to-nearest-even).  The sum is Neumaier-compensated (Neumaier 1974),
 *   so s carries far less than one fp32 ulp of error even for rows of 2^22
 *   terms; x_j - m is exact in binary64 for fp16/bf16/fp32 inputs whose
 *   exponents are within 2^52 of each other, which holds for every finite
 *   input that does not underflow exp.
 *
 *   the chunked online softmax: the running pair (m, d) updated chunk by chunk,
 *       m_new = max(m, max(chunk))
 *       d     = d * exp(m - m_new) + sum_{j in chunk} exp(x_j - m_new)
 *       m     = m_new
 *   followed by y_j = exp(x_j - m) / d, as stated in "[CUDA] safe online
 *   softmax", section 1, the safe_online_softmax listing (the per-element
 *   form of the same update is section 4.3 of "Softmax on DCU").  It equals
 *   the definition algebraically; the oracle keeps it as a self-check of the
 *   (m, d) rescaling rule that the split-k and streaming kernels rely on.
 *
 *   dtype decode (fp16, bf16, fp32 -> binary64, exact) and encode (binary64
 *   -> fp16 / bf16 / fp32, round to nearest, ties to even, straight from the
 *   binary64 value with no intermediate fp32 rounding), written from the
 *   IEEE 754-2008 binary16 layout and the bfloat16 layout (the top 16 bits of
 *   a binary32).  Round-to-nearest-even output is what "Softmax on DCU"
 *   section 4.5 and the "[CUDA] safe online softmax" kernels use when they
 *   write half results.
 *
 *   LayerNorm and RMSNorm along the last dimension (the operators "Softmax
 *   on DCU", section 9, names as having the same read - reduce - normalise -
 *   write structure; the Pangu-Weather profile, section 3, standardises fp16
 *   rows with fp32 mean and variance): the definitions written out at
 *   oracle_norm_f64 below.
 *
 * Non-finite inputs follow IEEE propagation through the definition above:
 * a NaN anywhere in a row, a +inf in a row, or a row that is all -inf gives a
 * NaN row; -inf entries in an otherwise finite row give exact zeros.
 *
 * Parity pins (tests/test_oracle_pins.py): the worked example of the HIP
 * softmax tutorial, its printed 4-element output, closed forms (cols = 1,
 * constant rows, the two-element logistic, a single planted peak), row sums,
 * bitwise shift invariance on dyadic grids, online == direct, scipy's
 * softmax on random rows, exhaustive fp16/bf16 decode against numpy / bit
 * reinterpretation, and encode against ties constructed at every midpoint.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_F16 1
#define ORACLE_BF16 2

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

/* ------------------------------------------------------------------------ */
/* decode                                                                    */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32 pattern. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_f32_to_f64(float f) { return (double)f; }

/* ------------------------------------------------------------------------ */
/* encode: round to nearest, ties to even, directly from binary64             */
/* ------------------------------------------------------------------------ */

/* Round a >= 0 to the nearest multiple of q (a power of two), ties to even
 * multiple.  a / q is exact in binary64 because q is a power of two and the
 * quotient stays in range for every case used below. */
static double round_to_quantum(double a, double q)
{
    double n = a / q;
    double r = floor(n);
    double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    return r * q;
}

/* Generic encoder for a binary format with `fbits` fraction bits, exponent
 * bias `bias` and all-ones exponent `emax_field` reserved for inf/NaN.
 * Returns the bit pattern in the low (1 + ebits + fbits) bits. */
static uint32_t encode_binary(double v, int ebits, int fbits)
{
    int bias = (1 << (ebits - 1)) - 1;
    int emax_field = (1 << ebits) - 1;
    uint32_t sign = signbit(v) ? 1u : 0u;
    uint32_t signbit_pos = (uint32_t)(ebits + fbits);
    if (isnan(v))
        return (sign << signbit_pos) | ((uint32_t)emax_field << fbits) | (1u << (fbits - 1));
    double a = fabs(v);
    /* largest finite value and the rounding threshold above which RNE gives inf */
    double maxf = ldexp(2.0 - ldexp(1.0, -fbits), bias);
    double ovf = ldexp(2.0 - ldexp(1.0, -fbits - 1), bias);
    if (isinf(a) || a >= ovf)
        return (sign << signbit_pos) | ((uint32_t)emax_field << fbits);
    int min_exp = 1 - bias; /* exponent of the smallest normal */
    double q;
    if (a < ldexp(1.0, min_exp)) {
        q = ldexp(1.0, min_exp - fbits); /* subnormal quantum */
    } else {
        int k;
        frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
        q = ldexp(1.0, (k - 1) - fbits);
    }
    double R = round_to_quantum(a, q);
    if (R > maxf) /* cannot happen below ovf, kept as a guard */
        return (sign << signbit_pos) | ((uint32_t)emax_field << fbits);
    uint32_t bits;
    if (R < ldexp(1.0, min_exp)) {
        /* subnormal (or zero): the fraction field counts quanta; a value that
         * rounded up to exactly the smallest normal gives 1 << fbits, which is
         * that normal's pattern. */
        bits = (uint32_t)(R / ldexp(1.0, min_exp - fbits));
    } else {
        int k;
        double f = frexp(R, &k);            /* R = f * 2^k, f in [0.5, 1) */
        int E = k - 1;                      /* R = (2f) * 2^E, 2f in [1, 2) */
        uint32_t frac = (uint32_t)((2.0 * f - 1.0) * ldexp(1.0, fbits));
        bits = ((uint32_t)(E + bias) << fbits) | frac;
    }
    return (sign << signbit_pos) | bits;
}

uint16_t oracle_f64_to_f16(double v) { return (uint16_t)encode_binary(v, 5, 10); }
uint16_t oracle_f64_to_bf16(double v) { return (uint16_t)encode_binary(v, 8, 7); }
float oracle_f64_to_f32(double v) { return (float)v; /* C conversion: RNE */ }

/* ------------------------------------------------------------------------ */
/* bulk decode / encode                                                       */
/* ------------------------------------------------------------------------ */

static double decode_at(const void *x, int dtype, int64_t i)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)x)[i];
    if (dtype == ORACLE_F16)
        return oracle_f16_to_f64(((const uint16_t *)x)[i]);
    return oracle_bf16_to_f64(((const uint16_t *)x)[i]);
}

int oracle_decode(const void *x, int dtype, int64_t n, double *out)
{
    if (n < 0 || dtype < 0 || dtype > 2 || (n > 0 && (!x || !out)))
        return ORACLE_EINVAL;
    for (int64_t i = 0; i < n; i++)
        out[i] = decode_at(x, dtype, i);
    return ORACLE_OK;
}

int oracle_encode(const double *y, int dtype, int64_t n, void *out)
{
    if (n < 0 || dtype < 0 || dtype > 2 || (n > 0 && (!y || !out)))
        return ORACLE_EINVAL;
    for (int64_t i = 0; i < n; i++) {
        if (dtype == ORACLE_F32)
            ((float *)out)[i] = oracle_f64_to_f32(y[i]);
        else if (dtype == ORACLE_F16)
            ((uint16_t *)out)[i] = oracle_f64_to_f16(y[i]);
        else
            ((uint16_t *)out)[i] = oracle_f64_to_bf16(y[i]);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* the definition                                                             */
/* ------------------------------------------------------------------------ */

/* max over a row with NaN made sticky (a NaN input makes the row NaN). */
static double row_max(const double *xr, int64_t cols)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < cols; j++) {
        if (isnan(xr[j]))
            return NAN;
        if (xr[j] > m)
            m = xr[j];
    }
    return m;
}

/* Neumaier's compensated sum of exp(x_j - m). */
static double row_expsum(const double *xr, int64_t cols, double m)
{
    double s = 0.0, c = 0.0;
    for (int64_t j = 0; j < cols; j++) {
        double t = exp(xr[j] - m);
        double u = s + t;
        if (fabs(s) >= fabs(t))
            c += (s - u) + t;
        else
            c += (t - u) + s;
        s = u;
    }
    return s + c;
}

/* One row of the definition: m = max, s = sum exp(x - m), y = exp(x - m)/s. */
static void softmax_row(const double *xr, int64_t cols, double *yr)
{
    double m = row_max(xr, cols);
    double s = row_expsum(xr, cols, m);
    for (int64_t j = 0; j < cols; j++)
        yr[j] = exp(xr[j] - m) / s;
}

int oracle_softmax_f64(const double *x, int64_t rows, int64_t cols, double *y)
{
    if (rows < 0 || cols < 0 || (rows > 0 && cols > 0 && (!x || !y)))
        return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        softmax_row(x + r * cols, cols, y + r * cols);
    return ORACLE_OK;
}

/* decode a [rows, cols] array of `dtype` and apply the definition. */
int oracle_softmax(const void *x, int dtype, int64_t rows, int64_t cols, double *y)
{
    if (rows < 0 || cols < 0 || dtype < 0 || dtype > 2 || (rows > 0 && cols > 0 && (!x || !y)))
        return ORACLE_EINVAL;
    int failed = 0;
#pragma omp parallel
    {
        double *xs = (rows > 0 && cols > 0) ? (double *)malloc((size_t)cols * sizeof(double)) : NULL;
        if (rows > 0 && cols > 0 && !xs) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; r++) {
            if (!xs)
                continue;
            for (int64_t j = 0; j < cols; j++)
                xs[j] = decode_at(x, dtype, r * cols + j);
            softmax_row(xs, cols, y + r * cols);
        }
        free(xs);
    }
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* the chunked online form (self-check of the (m, d) rescaling rule)          */
/* ------------------------------------------------------------------------ */

int oracle_online_softmax_f64(const double *x, int64_t rows, int64_t cols, int64_t chunk, double *y)
{
    if (rows < 0 || cols < 0 || chunk <= 0 || (rows > 0 && cols > 0 && (!x || !y)))
        return ORACLE_EINVAL;
    for (int64_t r = 0; r < rows; r++) {
        const double *xr = x + r * cols;
        double m = -INFINITY, d = 0.0;
        for (int64_t i = 0; i < cols; i += chunk) {
            int64_t end = i + chunk < cols ? i + chunk : cols;
            double m_local = row_max(xr + i, end - i);
            double m_new = (isnan(m_local) || isnan(m)) ? NAN : (m_local > m ? m_local : m);
            double d_local = row_expsum(xr + i, end - i, m_new);
            /* scale of the history: exp(m - m_new); with no history (d == 0,
             * m == -inf) the term is zero. */
            double scale = (d == 0.0 && m == -INFINITY) ? 0.0 : exp(m - m_new);
            d = d * scale + d_local;
            m = m_new;
        }
        for (int64_t j = 0; j < cols; j++)
            y[r * cols + j] = exp(xr[j] - m) / d;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* streaming comparison of a candidate output against the definition         */
/* ------------------------------------------------------------------------ */

/* Per-call summary of oracle_check.  Counts are over the rows checked. */
typedef struct {
    int64_t checked;           /* elements compared */
    int64_t violations;        /* elements outside the tolerance */
    int64_t nonfinite;         /* inf / NaN outputs on rows whose input is finite */
    int64_t first_bad;         /* flat index of the first violation, or -1 */
    double max_rel;            /* fp32: max |y - y*| / y* over y* >= abs_floor */
    int64_t max_ulp;           /* fp16 / bf16: max |bits(y) - bits(RNE(y*))| */
    double max_rowsum_dev;     /* max |sum_j y_j - 1| over finite-input rows */
    int64_t rowsum_violations; /* rows whose sum misses rowsum_a + cols * rowsum_b */
} oracle_check_result;

static int row_is_finite(const double *xr, int64_t cols)
{
    for (int64_t j = 0; j < cols; j++)
        if (!isfinite(xr[j]))
            return 0;
    return 1;
}

/* Tolerance parameters of a forward comparison. */
typedef struct {
    double rel_tol, abs_floor;
    int64_t max_ulp;
    double rowsum_a, rowsum_b;
    double zrel; /* masked form: extra relative allowance zrel * max_j |z_j| */
} oracle_tol;

/* Compare row r of a candidate output y with the wanted row `want`:
 *   fp32:        |y - y*| <= rel_tol * y* + abs_floor (+ zrel * zmax * y*)
 *   fp16, bf16:  |bits(y) - bits(RNE_dtype(y*))| <= max_ulp (outputs are >= 0,
 *                so the bit distance is the distance in ulps, subnormals and
 *                zero included), or |y - y*| <= zrel * zmax * y*; a NaN
 *                matches only a NaN.
 *   row sums:    |sum_j y_j - 1| <= rowsum_a + cols * rowsum_b on rows with
 *                finite inputs, y_j decoded exactly and summed in binary64. */
static void compare_row(const double *want, const void *y, int dtype, int64_t r, int64_t cols, int finite_row,
                        double zmax, const oracle_tol *t, oracle_check_result *loc)
{
    double s = 0.0, c = 0.0;
    for (int64_t j = 0; j < cols; j++) {
        int64_t flat = r * cols + j;
        double w = want[j];
        double got = decode_at(y, dtype, flat);
        double zallow = t->zrel * zmax * fabs(w);
        int bad = 0;
        if (finite_row && !isfinite(got))
            loc->nonfinite++;
        if (dtype == ORACLE_F32) {
            if (isnan(w) || isnan(got)) {
                bad = !(isnan(w) && isnan(got));
            } else {
                double err = fabs(got - w);
                bad = !(err <= t->rel_tol * fabs(w) + t->abs_floor + zallow);
                if (fabs(w) >= t->abs_floor && w != 0.0 && err / fabs(w) > loc->max_rel)
                    loc->max_rel = err / fabs(w);
            }
        } else {
            uint16_t gb = ((const uint16_t *)y)[flat];
            uint16_t wb = dtype == ORACLE_F16 ? oracle_f64_to_f16(w) : oracle_f64_to_bf16(w);
            if (isnan(w) || isnan(got)) {
                bad = !(isnan(w) && isnan(got));
            } else if ((gb | wb) & 0x8000u) {
                bad = gb != wb; /* a negative output matches only exactly */
            } else {
                int64_t dist = gb > wb ? (int64_t)gb - wb : (int64_t)wb - gb;
                if (dist > loc->max_ulp)
                    loc->max_ulp = dist;
                bad = dist > t->max_ulp && !(fabs(got - w) <= zallow);
            }
        }
        if (bad) {
            if (loc->first_bad < 0 || flat < loc->first_bad)
                loc->first_bad = flat;
            loc->violations++;
        }
        loc->checked++;
        if (finite_row) {
            double u = s + got;
            if (fabs(s) >= fabs(got))
                c += (s - u) + got;
            else
                c += (got - u) + s;
            s = u;
        }
    }
    if (finite_row) {
        double dev = fabs((s + c) - 1.0);
        if (!(dev <= t->rowsum_a + (double)cols * t->rowsum_b))
            loc->rowsum_violations++;
        if (dev > loc->max_rowsum_dev || isnan(dev))
            loc->max_rowsum_dev = isnan(dev) ? INFINITY : dev;
    }
}

static void merge_result(oracle_check_result *res, const oracle_check_result *loc)
{
    res->checked += loc->checked;
    res->violations += loc->violations;
    res->nonfinite += loc->nonfinite;
    res->rowsum_violations += loc->rowsum_violations;
    if (loc->first_bad >= 0 && (res->first_bad < 0 || loc->first_bad < res->first_bad))
        res->first_bad = loc->first_bad;
    if (loc->max_rel > res->max_rel)
        res->max_rel = loc->max_rel;
    if (loc->max_ulp > res->max_ulp)
        res->max_ulp = loc->max_ulp;
    if (loc->max_rowsum_dev > res->max_rowsum_dev)
        res->max_rowsum_dev = loc->max_rowsum_dev;
}

/* Compare y (same dtype and layout as x) with the definition applied to x
 * (compare_row gives the tolerances).  rows_sel (length n_sel) picks rows to
 * check; NULL checks all rows. */
int oracle_check(const void *x, const void *y, int dtype, int64_t rows, int64_t cols,
                 const int64_t *rows_sel, int64_t n_sel, double rel_tol, double abs_floor,
                 int64_t max_ulp, double rowsum_a, double rowsum_b, oracle_check_result *res)
{
    if (!res || rows < 0 || cols < 0 || dtype < 0 || dtype > 2)
        return ORACLE_EINVAL;
    memset(res, 0, sizeof *res);
    res->first_bad = -1;
    if (rows == 0 || cols == 0)
        return ORACLE_OK;
    if (!x || !y)
        return ORACLE_EINVAL;
    int64_t n = rows_sel ? n_sel : rows;
    for (int64_t i = 0; rows_sel && i < n; i++)
        if (rows_sel[i] < 0 || rows_sel[i] >= rows)
            return ORACLE_EINVAL;
    const oracle_tol tol = {rel_tol, abs_floor, max_ulp, rowsum_a, rowsum_b, 0.0};
    int failed = 0;
#pragma omp parallel
    {
        double *xs = (double *)malloc((size_t)cols * sizeof(double));
        double *ys = (double *)malloc((size_t)cols * sizeof(double));
        oracle_check_result loc;
        memset(&loc, 0, sizeof loc);
        loc.first_bad = -1;
        if (!xs || !ys) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < n; i++) {
            if (!xs || !ys)
                continue;
            int64_t r = rows_sel ? rows_sel[i] : i;
            for (int64_t j = 0; j < cols; j++)
                xs[j] = decode_at(x, dtype, r * cols + j);
            softmax_row(xs, cols, ys);
            compare_row(ys, y, dtype, r, cols, row_is_finite(xs, cols), 0.0, &tol, &loc);
        }
#pragma omp critical
        merge_result(res, &loc);
        free(xs);
        free(ys);
    }
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* scaled, masked softmax (attention scores)                                  */
/* ------------------------------------------------------------------------ */

/* The logits of row r:  z_j = scale * x_j + mask[r % mask_rows, j]  (mask may
 * be absent), and with a causal mask (causal_q > 0) z_j = -inf for every key
 * j > i + (cols - causal_q), i = r % causal_q the query index of the row (the
 * query block is aligned to the end of the keys).  The scaled, additively
 * masked softmax of "Softmax on DCU", section 9 (attention scores with scale
 * and mask fused into the softmax) and the bias + mask + softmax fusion of the
 * Pangu-Weather profile, section 6.  Binary64: scale * x is exact (24 x 24
 * bits), the sum with the mask rounds once. */
static void masked_logits(const void *x, const void *mask, int dtype, int64_t r, int64_t cols, double scale,
                          int64_t mask_rows, int64_t causal_q, double *z)
{
    int64_t limit = cols; /* keys j < limit are visible */
    if (causal_q > 0)
        limit = r % causal_q + (cols - causal_q) + 1;
    for (int64_t j = 0; j < cols; j++) {
        double v = scale * decode_at(x, dtype, r * cols + j);
        if (mask)
            v += decode_at(mask, dtype, (r % mask_rows) * cols + j);
        z[j] = j < limit ? v : -INFINITY;
    }
}

int oracle_softmax_masked(const void *x, int dtype, int64_t rows, int64_t cols, double scale, const void *mask,
                          int64_t mask_rows, int64_t causal_q, double *y)
{
    if (rows < 0 || cols < 0 || dtype < 0 || dtype > 2 || causal_q < 0 || (mask && mask_rows < 1) ||
        (rows > 0 && cols > 0 && (!x || !y)))
        return ORACLE_EINVAL;
    int failed = 0;
#pragma omp parallel
    {
        double *z = (rows > 0 && cols > 0) ? (double *)malloc((size_t)cols * sizeof(double)) : NULL;
        if (rows > 0 && cols > 0 && !z) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; r++) {
            if (!z)
                continue;
            masked_logits(x, mask, dtype, r, cols, scale, mask_rows, causal_q, z);
            softmax_row(z, cols, y + r * cols);
        }
        free(z);
    }
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}

/* Compare a candidate with the masked definition; the tolerances of
 * compare_row, plus zrel * max_j |z_j| relative (the rounding of the logits
 * themselves in fp32). */
int oracle_check_masked(const void *x, const void *y, int dtype, int64_t rows, int64_t cols, double scale,
                        const void *mask, int64_t mask_rows, int64_t causal_q, double rel_tol, double abs_floor,
                        int64_t max_ulp, double rowsum_a, double rowsum_b, double zrel, oracle_check_result *res)
{
    if (!res || rows < 0 || cols < 0 || dtype < 0 || dtype > 2 || causal_q < 0 || (mask && mask_rows < 1))
        return ORACLE_EINVAL;
    memset(res, 0, sizeof *res);
    res->first_bad = -1;
    if (rows == 0 || cols == 0)
        return ORACLE_OK;
    if (!x || !y)
        return ORACLE_EINVAL;
    const oracle_tol tol = {rel_tol, abs_floor, max_ulp, rowsum_a, rowsum_b, zrel};
    int failed = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc((size_t)cols * sizeof(double));
        double *ys = (double *)malloc((size_t)cols * sizeof(double));
        oracle_check_result loc;
        memset(&loc, 0, sizeof loc);
        loc.first_bad = -1;
        if (!z || !ys) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; r++) {
            if (!z || !ys)
                continue;
            masked_logits(x, mask, dtype, r, cols, scale, mask_rows, causal_q, z);
            double zmax = 0.0;
            int finite = 1;
            for (int64_t j = 0; j < cols; j++) {
                if (isnan(z[j]) || z[j] == INFINITY)
                    finite = 0;
                else if (isfinite(z[j]) && fabs(z[j]) > zmax)
                    zmax = fabs(z[j]);
            }
            /* a row with no visible key is all -inf: finite inputs, NaN by the
             * definition; treat it as non-finite for the row-sum check */
            int any_visible = 0;
            for (int64_t j = 0; j < cols; j++)
                any_visible |= z[j] != -INFINITY;
            softmax_row(z, cols, ys);
            compare_row(ys, y, dtype, r, cols, finite && any_visible, zmax, &tol, &loc);
        }
#pragma omp critical
        merge_result(res, &loc);
        free(z);
        free(ys);
    }
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}

/* Number of OpenMP threads a parallel region of the oracle uses (1 without
 * OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of OpenMP threads later parallel regions started from the
 * calling host thread use (n >= 1; the CPU baseline times the oracle on all
 * cores and on one).  Returns the number in force afterwards. */
int oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* backward: dx = y * (dy - sum_k dy_k y_k)                                   */
/* ------------------------------------------------------------------------ */

/* The gradient of L(x) through y = softmax(x): dL/dx_j = sum_i dy_i dy_i/dx_j
 * with dy_i/dx_j = y_i (delta_ij - y_j), i.e. dx_j = y_j (dy_j - s), s = sum_k
 * dy_k y_k.  The pages name the backward pass as separate work ("Softmax on
 * DCU", section 5.4, accuracy validation beyond inference); the formula is
 * this derivative of the definition, written out. */
static void softmax_bwd_row(const double *yr, const double *dyr, int64_t cols, double *dxr)
{
    double s = 0.0, c = 0.0;
    for (int64_t j = 0; j < cols; j++) {
        double t = dyr[j] * yr[j];
        double u = s + t;
        if (fabs(s) >= fabs(t))
            c += (s - u) + t;
        else
            c += (t - u) + s;
        s = u;
    }
    s += c;
    for (int64_t j = 0; j < cols; j++)
        dxr[j] = yr[j] * (dyr[j] - s);
}

int oracle_softmax_bwd_f64(const double *y, const double *dy, int64_t rows, int64_t cols, double *dx)
{
    if (rows < 0 || cols < 0 || (rows > 0 && cols > 0 && (!y || !dy || !dx)))
        return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        softmax_bwd_row(y + r * cols, dy + r * cols, cols, dx + r * cols);
    return ORACLE_OK;
}

/* spacing of the dtype at |v| (the ulp a value of that magnitude has) */
static double dtype_ulp(double v, int dtype)
{
    int fbits = dtype == ORACLE_F32 ? 23 : (dtype == ORACLE_F16 ? 10 : 7);
    int min_exp = dtype == ORACLE_F32 ? -126 : (dtype == ORACLE_F16 ? -14 : -126);
    double a = fabs(v);
    int k;
    if (a == 0.0 || !isfinite(a))
        return ldexp(1.0, min_exp - fbits);
    frexp(a, &k);
    int e = k - 1;
    if (e < min_exp)
        e = min_exp;
    return ldexp(1.0, e - fbits);
}

/* Compare a candidate dx (dtype) with the backward definition applied to the
 * decoded y and dy.  Element j passes when
 *     |dx_j - dx*_j| <= max_ulp * ulp_dtype(dx*_j) + rel_tol * |dx*_j|
 *                       + k_eps * 2^-24 * |y_j| * (|dy_j| + sum_k |dy_k y_k|)
 * The last term is the fp32 cancellation budget of dy_j - s: it is the
 * error an fp32 evaluation of s and of the difference carries relative to the
 * magnitudes involved, which can exceed any relative bound on dx*_j when the
 * difference nearly cancels. */
int oracle_check_bwd(const void *y, const void *dy, const void *dx, int dtype, int64_t rows, int64_t cols,
                     double rel_tol, int64_t max_ulp, double k_eps, oracle_check_result *res)
{
    if (!res || rows < 0 || cols < 0 || dtype < 0 || dtype > 2)
        return ORACLE_EINVAL;
    memset(res, 0, sizeof *res);
    res->first_bad = -1;
    if (rows == 0 || cols == 0)
        return ORACLE_OK;
    if (!y || !dy || !dx)
        return ORACLE_EINVAL;
    int failed = 0;
#pragma omp parallel
    {
        double *ys = (double *)malloc((size_t)cols * sizeof(double));
        double *dys = (double *)malloc((size_t)cols * sizeof(double));
        double *want = (double *)malloc((size_t)cols * sizeof(double));
        oracle_check_result loc;
        memset(&loc, 0, sizeof loc);
        loc.first_bad = -1;
        if (!ys || !dys || !want) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; r++) {
            if (!ys || !dys || !want)
                continue;
            double sabs = 0.0;
            for (int64_t j = 0; j < cols; j++) {
                ys[j] = decode_at(y, dtype, r * cols + j);
                dys[j] = decode_at(dy, dtype, r * cols + j);
                sabs += fabs(ys[j] * dys[j]);
            }
            softmax_bwd_row(ys, dys, cols, want);
            for (int64_t j = 0; j < cols; j++) {
                int64_t flat = r * cols + j;
                double got = decode_at(dx, dtype, flat);
                double w = want[j];
                int bad;
                if (isnan(w) || isnan(got)) {
                    bad = !(isnan(w) && isnan(got));
                } else {
                    double err = fabs(got - w);
                    double bound = (double)max_ulp * dtype_ulp(w, dtype) + rel_tol * fabs(w) +
                                   k_eps * ldexp(1.0, -24) * fabs(ys[j]) * (fabs(dys[j]) + sabs);
                    bad = !(err <= bound);
                    if (!isfinite(got))
                        loc.nonfinite++;
                    double ulps = err / dtype_ulp(w, dtype);
                    if ((int64_t)ulps > loc.max_ulp)
                        loc.max_ulp = (int64_t)ulps;
                    if (w != 0.0 && err / fabs(w) > loc.max_rel)
                        loc.max_rel = err / fabs(w);
                }
                if (bad) {
                    if (loc.first_bad < 0 || flat < loc.first_bad)
                        loc.first_bad = flat;
                    loc.violations++;
                }
                loc.checked++;
            }
        }
#pragma omp critical
        {
            res->checked += loc.checked;
            res->violations += loc.violations;
            res->nonfinite += loc.nonfinite;
            if (loc.first_bad >= 0 && (res->first_bad < 0 || loc.first_bad < res->first_bad))
                res->first_bad = loc.first_bad;
            if (loc.max_rel > res->max_rel)
                res->max_rel = loc.max_rel;
            if (loc.max_ulp > res->max_ulp)
                res->max_ulp = loc.max_ulp;
        }
        free(ys);
        free(dys);
        free(want);
    }
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* LayerNorm and RMSNorm along the last dimension                             */
/* ------------------------------------------------------------------------ */

/* "Softmax on DCU", section 9, names LayerNorm and RMSNorm as operators with
 * the softmax's read - reduce - normalise - write structure; the Pangu-Weather
 * profile, section 3, standardises fp16 rows with fp32 mean and variance (its
 * affine parameters folded into the next layer).  Written out, per row of n
 * values x_j, with optional per-column gain g_j and bias b_j (absent: g = 1,
 * b = 0):
 *   LayerNorm:  mu   = (1/n) sum_j x_j
 *               var  = (1/n) sum_j (x_j - mu)^2      (population variance,
 *                                                      about the mean: two passes)
 *               rstd = 1 / sqrt(var + eps)
 *               y_j  = (x_j - mu) * rstd * g_j + b_j
 *   RMSNorm:    ms   = (1/n) sum_j x_j^2
 *               rstd = 1 / sqrt(ms + eps)
 *               y_j  = x_j * rstd * g_j                (no bias)
 * Binary64 throughout; the sums are Neumaier-compensated. */

#define ORACLE_LAYERNORM 0
#define ORACLE_RMSNORM 1

static double nsum_add(double s, double t, double *c)
{
    double u = s + t;
    if (fabs(s) >= fabs(t))
        *c += (s - u) + t;
    else
        *c += (t - u) + s;
    return u;
}

/* One row: y (n values), and the statistics mu (LayerNorm; 0 for RMSNorm),
 * rstd and a = (1/n) sum_j |x_j| (the scale of the rounding errors an fp32
 * evaluation of the statistics makes). */
static void norm_row(int kind, const double *x, int64_t n, const double *g, const double *b, double eps,
                     double *y, double *mu_out, double *rstd_out, double *a_out)
{
    double s = 0.0, c = 0.0, sa = 0.0, ca = 0.0;
    for (int64_t j = 0; j < n; j++) {
        s = nsum_add(s, x[j], &c);
        sa = nsum_add(sa, fabs(x[j]), &ca);
    }
    const double mu = kind == ORACLE_LAYERNORM ? (s + c) / (double)n : 0.0;
    double q = 0.0, cq = 0.0;
    for (int64_t j = 0; j < n; j++) {
        double d = x[j] - mu;
        q = nsum_add(q, d * d, &cq);
    }
    const double var = (q + cq) / (double)n;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int64_t j = 0; j < n; j++) {
        double v = (x[j] - mu) * rstd;
        if (g)
            v *= g[j];
        if (b && kind == ORACLE_LAYERNORM)
            v += b[j];
        y[j] = v;
    }
    *mu_out = mu;
    *rstd_out = rstd;
    *a_out = (sa + ca) / (double)n;
}

static int decode_vec(const void *v, int dtype, int64_t n, double **out)
{
    *out = NULL;
    if (!v)
        return 0;
    *out = (double *)malloc((size_t)n * sizeof(double));
    if (!*out)
        return -1;
    for (int64_t j = 0; j < n; j++)
        (*out)[j] = decode_at(v, dtype, j);
    return 0;
}

/* y (binary64, [rows, cols]) = the norm of x (dtype); gamma, beta: [cols] in
 * x's dtype or NULL; mean, rstd: [rows] binary64 or NULL. */
int oracle_norm_f64(int kind, const void *x, int dtype, int64_t rows, int64_t cols, const void *gamma,
                    const void *beta, double eps, double *y, double *mean, double *rstd)
{
    if ((kind != ORACLE_LAYERNORM && kind != ORACLE_RMSNORM) || rows < 0 || cols < 0 || dtype < 0 ||
        dtype > 2 || !(eps >= 0.0) || (rows > 0 && cols > 0 && (!x || !y)))
        return ORACLE_EINVAL;
    if (rows == 0 || cols == 0)
        return ORACLE_OK;
    double *g = NULL, *b = NULL;
    if (decode_vec(gamma, dtype, cols, &g) || decode_vec(beta, dtype, cols, &b)) {
        free(g);
        free(b);
        return ORACLE_EINVAL;
    }
    int failed = 0;
#pragma omp parallel
    {
        double *xs = (double *)malloc((size_t)cols * sizeof(double));
        if (!xs) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; r++) {
            if (!xs)
                continue;
            for (int64_t j = 0; j < cols; j++)
                xs[j] = decode_at(x, dtype, r * cols + j);
            double mu, rs, a;
            norm_row(kind, xs, cols, g, b, eps, y + r * cols, &mu, &rs, &a);
            if (mean)
                mean[r] = mu;
            if (rstd)
                rstd[r] = rs;
        }
        free(xs);
    }
    free(g);
    free(b);
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}

/* Compare a candidate y (dtype) -- and, when given, its fp32 per-row mean and
 * rstd -- with the definition.  Element j passes when
 *     |y_j - y*_j| <= max_ulp * ulp_dtype(y*_j) + rel_tol * |y*_j|
 *                     + k_eps * 2^-24 * (|g_j| * (|z_j| + a * rstd) + |b_j|)
 * with z_j = (x_j - mu) * rstd the normalised value, a = (1/n) sum |x_j| and
 * the a * rstd term only for LayerNorm: fp32 statistics carry errors of a few
 * 2^-24 relative to the magnitudes summed, and an error d in mu moves every
 * output by d * rstd * g_j, which no relative bound on y*_j covers where
 * x_j is close to mu.  The statistics pass when |mean - mu| <= k_eps * 2^-24 *
 * a and |rstd - rstd*| <= k_eps * 2^-24 * rstd*. */
int oracle_check_norm(int kind, const void *x, const void *y, int dtype, int64_t rows, int64_t cols,
                      const void *gamma, const void *beta, double eps, const float *mean, const float *rstd,
                      double rel_tol, int64_t max_ulp, double k_eps, oracle_check_result *res)
{
    if (!res || (kind != ORACLE_LAYERNORM && kind != ORACLE_RMSNORM) || rows < 0 || cols < 0 || dtype < 0 ||
        dtype > 2 || !(eps >= 0.0))
        return ORACLE_EINVAL;
    memset(res, 0, sizeof *res);
    res->first_bad = -1;
    if (rows == 0 || cols == 0)
        return ORACLE_OK;
    if (!x || !y)
        return ORACLE_EINVAL;
    double *g = NULL, *b = NULL;
    if (decode_vec(gamma, dtype, cols, &g) || decode_vec(beta, dtype, cols, &b)) {
        free(g);
        free(b);
        return ORACLE_EINVAL;
    }
    const double u = k_eps * ldexp(1.0, -24);
    int failed = 0;
#pragma omp parallel
    {
        double *xs = (double *)malloc((size_t)cols * sizeof(double));
        double *want = (double *)malloc((size_t)cols * sizeof(double));
        oracle_check_result loc;
        memset(&loc, 0, sizeof loc);
        loc.first_bad = -1;
        if (!xs || !want) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; r++) {
            if (!xs || !want)
                continue;
            for (int64_t j = 0; j < cols; j++)
                xs[j] = decode_at(x, dtype, r * cols + j);
            double mu, rs, a;
            norm_row(kind, xs, cols, g, b, eps, want, &mu, &rs, &a);
            const double shift = kind == ORACLE_LAYERNORM ? a * rs : 0.0;
            for (int64_t j = 0; j < cols; j++) {
                int64_t flat = r * cols + j;
                double got = decode_at(y, dtype, flat);
                double w = want[j];
                int bad;
                if (isnan(w) || isnan(got)) {
                    bad = !(isnan(w) && isnan(got));
                } else {
                    double z = (xs[j] - mu) * rs;
                    double gj = g ? fabs(g[j]) : 1.0;
                    double bj = (b && kind == ORACLE_LAYERNORM) ? fabs(b[j]) : 0.0;
                    double err = fabs(got - w);
                    double bound = (double)max_ulp * dtype_ulp(w, dtype) + rel_tol * fabs(w) +
                                   u * (gj * (fabs(z) + shift) + bj);
                    bad = !(err <= bound);
                    if (!isfinite(got))
                        loc.nonfinite++;
                    double ulps = err / dtype_ulp(w, dtype);
                    if ((int64_t)ulps > loc.max_ulp)
                        loc.max_ulp = (int64_t)ulps;
                    if (w != 0.0 && err / fabs(w) > loc.max_rel)
                        loc.max_rel = err / fabs(w);
                }
                if (bad) {
                    if (loc.first_bad < 0 || flat < loc.first_bad)
                        loc.first_bad = flat;
                    loc.violations++;
                }
                loc.checked++;
            }
            /* the statistics (their violations count in rowsum_violations) */
            int sbad = 0;
            if (mean && kind == ORACLE_LAYERNORM && isfinite(mu))
                sbad |= !(fabs((double)mean[r] - mu) <= u * a);
            if (rstd && isfinite(rs))
                sbad |= !(fabs((double)rstd[r] - rs) <= u * rs);
            if (sbad)
                loc.rowsum_violations++;
        }
#pragma omp critical
        merge_result(res, &loc);
        free(xs);
        free(want);
    }
    free(g);
    free(b);
    return failed ? ORACLE_EINVAL : ORACLE_OK;
}
