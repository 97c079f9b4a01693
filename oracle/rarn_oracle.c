/*
 * rarn_oracle.c -- plain CPU oracle for row-wise RMSNorm and its fused
 * residual-add / reduce + residual-add forms.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * compared against.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.  It
 * shares no code, header, table or helper with the CUDA sources.
 *
 * What it computes (per row t of a row-major [T, H] problem):
 *
 *   1. h  -- the row that is normalised.
 *        plain:   h_i = x_i
 *        fused:   h_i = RN_dt( fl32( x_i + r_i ) )
 *        reduce:  acc = p0_i; acc = fl32(acc + p1_i); ... ; acc = fl32(acc + p{R-1}_i);
 *                 acc = fl32(acc + r_i);  h_i = RN_dt(acc)
 *      "Tokenweave fused-RMSNorm-AR kernel", Code walkthrough: the first
 *      pass reduces the partial buffers, adds the residual, stores the sum
 *      back as the new residual and accumulates the squares of that stored
 *      value.  The pages leave the order of the partial sum to the hardware;
 *      this oracle fixes it to p0, p1, ..., p{R-1}, then the residual, each
 *      add in binary32, and rounds once to the storage type.
 *   2. ss = sum_i h_i^2                     (binary64, index order)
 *   3. inv = 1 / sqrt(ss / H + eps)         (binary64; eps is the binary32
 *                                            argument widened)
 *      "RMSNorm kernel", 1 Background and 2 Analytics & Implementation
 *      (Abstraction): RMS over the last dimension only, mean of the squares
 *      plus eps under the root; the tokenweave kernel divides by the full
 *      hidden size before adding eps.
 *   4. y_i = RN_dt( (h_i * inv) * gamma_i )  (binary64 product, one rounding)
 *      "RMSNorm kernel", Abstraction step 2: elementwise x_i * gamma_i / RMS.
 *
 * Storage types: binary32 (f32), binary16 (f16), bfloat16 (bf16).  RN_dt is
 * round-to-nearest-even into the storage type, with IEEE overflow to
 * infinity and gradual underflow; it is written from the formats'
 * definitions (precision p, minimum exponent emin, maximum exponent emax).
 *
 * 8-bit output (oracle_rows_fp8): steps 1-3, then v_i = (h_i * inv) * gamma_i
 * in binary64 and the code q_i = FP8( v_i / s ), FP8 being nearest-even
 * rounding to e4m3 or e5m2 with saturation to the largest finite value
 * ("Block All Reduce", FP8 section: both formats, saturating conversion).
 * s is a given per-tensor binary32 scale, or per row max_i |v_i| / maxf, so
 * that the row's largest magnitude maps to the format's largest value.  The
 * pages give no formula for the scale; this is the plainest reading of a
 * per-row (dynamic) scale.
 *
 * 8-bit partials (oracle_reduce_fp8in): the reduce form with each partial
 * given as e4m3 / e5m2 codes c_r and a binary32 scale s_r per partial buffer
 * ("Block All Reduce", FP8 section: reductions over 8-bit inputs with a
 * binary32 accumulator).  Its value enters the sum as fl32(dec(c_r) * s_r),
 * one binary32 rounding of the product; then acc = that value for r = 0,
 * acc = fl32(acc + fl32(dec(c_r) * s_r)) for r = 1 .. R-1, acc = fl32(acc +
 * r_i), h_i = RN_dt(acc), and steps 2-4 as above.  The pages fix no scale
 * rule; a per-buffer (per-tensor) scale is the plainest reading.
 *
 * Tensor-parallel form (oracle_tp_reduce_add_rms_norm): N ranks each hold a
 * partial [T, H] (the output of a row-parallel layer) and the residual rows
 * of their own block of tokens; "Tokenweave fused-RMSNorm-AR kernel", Code
 * walkthrough: each rank reduces its tokens' rows over every rank's buffer
 * (the reduce-scatter), adds its residual, stores it, normalises, and writes
 * the normalised row into every rank's buffer (the all-gather).  Readings:
 * rank r owns rows floor(r T / N) .. floor((r + 1) T / N) - 1 (contiguous,
 * in rank order); the partials are summed in rank order 0 .. N-1 in binary32
 * (the pages leave the order to the switch's multimem reduction), then the
 * residual, one rounding -- the reduce form with R = N.
 *
 * Build flags must keep binary32 arithmetic exact IEEE: no -ffast-math, and
 * -ffp-contract=off (there is no multiply in the binary32 part, but the flag
 * documents the intent).
 */
#define _POSIX_C_SOURCE 200809L
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ----------------------------------------------------------------------- */
/* Storage formats                                                          */
/* ----------------------------------------------------------------------- */

static int elem_size(int dt) { return dt == ORC_F32 ? 4 : 2; }

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t b) {
    int sign = b >> 15;
    int e = (b >> 10) & 0x1f;
    int m = b & 0x3ff;
    double v;
    if (e == 0x1f) {
        v = m ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -24);          /* subnormal: m * 2^-24 */
    } else {
        v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32 pattern. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double load_elem(int dt, const void *base, int64_t i) {
    if (dt == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    }
    uint16_t b = ((const uint16_t *)base)[i];
    return dt == ORC_F16 ? half_bits_to_double(b) : bf16_bits_to_double(b);
}

/*
 * Round v to the nearest value of a binary format with p significand bits,
 * normal exponents emin..emax, ties to even.  Returns the rounded value as a
 * double (exact: every such format is a subset of binary64 here).
 */
static double round_to_format(double v, int p, int emin, int emax) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int e2;
    frexp(fabs(v), &e2);          /* |v| = m * 2^e2, m in [0.5, 1) */
    int lead = e2 - 1;            /* exponent of the leading bit */
    if (lead < emin) lead = emin; /* below the normal range the quantum is fixed */
    int q = lead - (p - 1);       /* exponent of one unit in the last place */
    double r = nearbyint(ldexp(v, -q)); /* default mode: nearest, ties to even */
    double out = ldexp(r, q);
    double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(out) > max_finite) return copysign(INFINITY, v);
    return out;
}

static double round_dt(int dt, double v) {
    switch (dt) {
    case ORC_F32: return round_to_format(v, 24, -126, 127);
    case ORC_F16: return round_to_format(v, 11, -14, 15);
    default: return round_to_format(v, 8, -126, 127);
    }
}

/* Encode a value that is already exactly representable in dt. */
static void store_exact(int dt, void *base, int64_t i, double v) {
    if (dt == ORC_F32) {
        float f = (float)v;
        memcpy((char *)base + 4 * i, &f, 4);
        return;
    }
    uint16_t b;
    if (dt == ORC_BF16) {
        float f = (float)v; /* exact: v has at most 8 significant bits */
        uint32_t u;
        memcpy(&u, &f, 4);
        b = (uint16_t)(u >> 16);
        if (isnan(v)) b = 0x7fc0;
    } else {
        uint16_t s = signbit(v) ? 0x8000 : 0;
        double a = fabs(v);
        if (isnan(v)) {
            b = 0x7e00;
        } else if (isinf(a)) {
            b = s | 0x7c00;
        } else if (a == 0.0) {
            b = s;
        } else {
            int e2;
            frexp(a, &e2);
            int lead = e2 - 1;
            if (lead >= -14) {
                int frac = (int)ldexp(a, 10 - lead) - 1024;
                b = s | (uint16_t)((lead + 15) << 10) | (uint16_t)frac;
            } else {
                b = s | (uint16_t)ldexp(a, 24);
            }
        }
    }
    ((uint16_t *)base)[i] = b;
}

/* ----------------------------------------------------------------------- */
/* One row                                                                  */
/* ----------------------------------------------------------------------- */

typedef struct {
    int dt;                    /* storage type of x / partials, gamma and y */
    int rdt;                   /* storage type of the residual (in and out) */
    int64_t T, H;
    int32_t R;                 /* number of partial buffers; 0 = plain */
    const void *x;             /* plain: x; fused/reduce: partials (R buffers) */
    int64_t ldx;               /* elements between rows of x / of each partial */
    int64_t slice;             /* elements between partial buffers */
    const void *residual_in;   /* or NULL (plain) */
    int64_t ldr;               /* elements between rows of the residual (in and out) */
    const void *gamma;         /* [H] */
    float eps;
    void *residual_out;        /* or NULL */
    void *y;
    int64_t ldy;               /* elements between rows of y */
    double *inv_out;           /* [T] or NULL */
    double *y64_out;           /* [T, H] dense or NULL: y before the final rounding */
} job_t;

static void one_row(const job_t *j, int64_t t, double *h) {
    const int64_t H = j->H;
    const int64_t xrow = t * j->ldx;
    const int64_t rrow = t * j->ldr;
    const int64_t yrow = t * j->ldy;

    /* step 1: h */
    if (j->residual_in == NULL) {
        for (int64_t i = 0; i < H; ++i) h[i] = load_elem(j->dt, j->x, xrow + i);
    } else {
        for (int64_t i = 0; i < H; ++i) {
            float acc = (float)load_elem(j->dt, j->x, xrow + i);
            for (int32_t r = 1; r < j->R; ++r)
                acc = acc + (float)load_elem(j->dt, j->x, (int64_t)r * j->slice + xrow + i);
            acc = acc + (float)load_elem(j->rdt, j->residual_in, rrow + i);
            h[i] = round_dt(j->rdt, (double)acc);
        }
        if (j->residual_out)
            for (int64_t i = 0; i < H; ++i) store_exact(j->rdt, j->residual_out, rrow + i, h[i]);
    }

    /* step 2: sum of squares of the (stored) row */
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) ss += h[i] * h[i];

    /* step 3: reciprocal RMS */
    double inv = 1.0 / sqrt(ss / (double)H + (double)j->eps);
    if (j->inv_out) j->inv_out[t] = inv;

    /* step 4: scale, weight, one rounding */
    for (int64_t i = 0; i < H; ++i) {
        double v = (h[i] * inv) * load_elem(j->dt, j->gamma, i);
        if (j->y64_out) j->y64_out[t * H + i] = v;
        store_exact(j->dt, j->y, yrow + i, round_dt(j->dt, v));
    }
}

/* Rows are independent: a row function is run over row ranges in host
 * threads, each with its own scratch of `scratch` doubles. */
typedef void (*row_fn)(const void *ctx, int64_t t, double *scratch);

typedef struct {
    const void *ctx;
    row_fn fn;
    int64_t t0, t1, scratch;
    int rc;
} slice_t;

static void *worker(void *arg) {
    slice_t *s = (slice_t *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)(s->scratch > 0 ? s->scratch : 1));
    if (!h) {
        s->rc = -1;
        return NULL;
    }
    for (int64_t t = s->t0; t < s->t1; ++t) s->fn(s->ctx, t, h);
    free(h);
    s->rc = 0;
    return NULL;
}

/* Runs rows 0..T-1 over nthreads host threads (0 = every online core).
 * Returns the number of threads used, or a negative value on error. */
static int run_rows(const void *ctx, row_fn fn, int64_t T, int64_t scratch, int nthreads) {
    if (T == 0) return 0;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > T) nthreads = (int)T;
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *made = (char *)calloc((size_t)nthreads, 1);
    slice_t *sl = (slice_t *)calloc((size_t)nthreads, sizeof(slice_t));
    if (!tid || !made || !sl) {
        free(tid);
        free(made);
        free(sl);
        return -1;
    }
    int rc = nthreads;
    for (int k = 0; k < nthreads; ++k) {
        sl[k].ctx = ctx;
        sl[k].fn = fn;
        sl[k].t0 = T * k / nthreads;
        sl[k].t1 = T * (k + 1) / nthreads;
        sl[k].scratch = scratch;
        sl[k].rc = -1;
        if (nthreads > 1 && pthread_create(&tid[k], NULL, worker, &sl[k]) == 0)
            made[k] = 1;
        else
            worker(&sl[k]); /* one thread, or a thread could not be created: inline */
    }
    for (int k = 0; k < nthreads; ++k)
        if (made[k]) pthread_join(tid[k], NULL);
    for (int k = 0; k < nthreads; ++k)
        if (sl[k].rc != 0) rc = -1;
    free(tid);
    free(made);
    free(sl);
    return rc;
}

static void job_row(const void *ctx, int64_t t, double *h) { one_row((const job_t *)ctx, t, h); }

static int run(const job_t *j, int nthreads) {
    if (j->T < 0 || j->H <= 0 || !j->x || !j->gamma || !j->y) return -2;
    return run_rows(j, job_row, j->T, j->H, nthreads);
}

/* ----------------------------------------------------------------------- */
/* Exported entry points (ctypes)                                           */
/* ----------------------------------------------------------------------- */

int oracle_rms_norm(int dt, int64_t T, int64_t H, const void *x, const void *gamma, float eps,
                    void *y, double *inv_out, double *y64_out, int nthreads) {
    job_t j = {dt, dt, T, H, 0, x, H, T * H, NULL, H, gamma, eps, NULL, y, H, inv_out, y64_out};
    return run(&j, nthreads);
}

int oracle_fused_add_rms_norm(int dt, int64_t T, int64_t H, const void *x, const void *residual_in,
                              const void *gamma, float eps, void *residual_out, void *y,
                              double *inv_out, double *y64_out, int nthreads) {
    if (!residual_in) return -2;
    job_t j = {dt, dt, T, H, 1, x, H, T * H, residual_in, H, gamma, eps, residual_out, y, H,
               inv_out, y64_out};
    return run(&j, nthreads);
}

int oracle_reduce_add_rms_norm(int dt, int64_t T, int64_t H, int32_t R, const void *partials,
                               const void *residual_in, const void *gamma, float eps,
                               void *residual_out, void *y, double *inv_out, double *y64_out,
                               int nthreads) {
    if (!residual_in || R < 1) return -2;
    job_t j = {dt, dt, T, H, R, partials, H, T * H, residual_in, H, gamma, eps, residual_out, y, H,
               inv_out, y64_out};
    return run(&j, nthreads);
}

/*
 * General form: every buffer has its own row stride (in elements, >= H), the
 * partial buffers are `slice` elements apart, and the residual has its own
 * storage type `rdt` (the sum is rounded once to rdt, which is the identity
 * for binary32).  R = 0: plain (residual ignored); R >= 1: partials (x for
 * R = 1) plus residual.  The residual is updated in place (residual_out may
 * equal residual_in).  Only the first H elements of each row of y and of the
 * residual are written.
 */
int oracle_rows_ex(int dt, int rdt, int64_t T, int64_t H, int32_t R, const void *x, int64_t ldx,
                   int64_t slice, const void *residual_in, void *residual_out, int64_t ldr,
                   const void *gamma, float eps, void *y, int64_t ldy, double *inv_out,
                   double *y64_out, int nthreads) {
    if (R < 0 || ldx < H || ldy < H || (R >= 1 && (!residual_in || ldr < H))) return -2;
    job_t j = {dt, rdt, T, H, R, x, ldx, slice, R >= 1 ? residual_in : NULL, ldr, gamma, eps,
               R >= 1 ? residual_out : NULL, y, ldy, inv_out, y64_out};
    return run(&j, nthreads);
}

/* ----------------------------------------------------------------------- */
/* Tensor-parallel form: reduce-scatter, residual + norm, all-gather        */
/* ----------------------------------------------------------------------- */

/* Rows of rank r among N: [floor(r T / N), floor((r + 1) T / N)). */
void oracle_tp_rows(int64_t T, int32_t N, int32_t r, int64_t *r0, int64_t *r1) {
    *r0 = T * (int64_t)r / N;
    *r1 = T * (int64_t)(r + 1) / N;
}

typedef struct {
    int dt;
    int64_t H;
    int32_t N;
    const void *const *bufs; /* N partials [T, H] */
    const void *residual_in; /* [T, H]: the ranks' blocks of rows, stacked */
    void *residual_out;
    const void *gamma;
    float eps;
    void *const *y_out;      /* N outputs [T, H], one per rank */
    double *inv_out;
    double *y64_out;
} tp_job_t;

/* Row t, computed by the rank that owns it. */
static void tp_row(const void *ctx, int64_t t, double *h) {
    const tp_job_t *j = (const tp_job_t *)ctx;
    const int64_t H = j->H, row = t * H;
    /* reduce-scatter: this rank's row over every rank's buffer, rank order */
    for (int64_t i = 0; i < H; ++i) {
        float rank_sum = (float)load_elem(j->dt, j->bufs[0], row + i);
        for (int32_t q = 1; q < j->N; ++q)
            rank_sum = rank_sum + (float)load_elem(j->dt, j->bufs[q], row + i);
        rank_sum = rank_sum + (float)load_elem(j->dt, j->residual_in, row + i);
        h[i] = round_dt(j->dt, (double)rank_sum);
    }
    for (int64_t i = 0; i < H; ++i) store_exact(j->dt, j->residual_out, row + i, h[i]);
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) ss += h[i] * h[i];
    const double inv = 1.0 / sqrt(ss / (double)H + (double)j->eps);
    if (j->inv_out) j->inv_out[t] = inv;
    /* all-gather: the normalised row into every rank's buffer */
    for (int64_t i = 0; i < H; ++i) {
        const double v = (h[i] * inv) * load_elem(j->dt, j->gamma, i);
        if (j->y64_out) j->y64_out[row + i] = v;
        const double yv = round_dt(j->dt, v);
        for (int32_t q = 0; q < j->N; ++q) store_exact(j->dt, j->y_out[q], row + i, yv);
    }
}

/* Each rank's block of rows in turn (rows within a block over host threads).
 * Returns the threads used, or a negative value on error. */
int oracle_tp_reduce_add_rms_norm(int dt, int64_t T, int64_t H, int32_t N,
                                  const void *const *bufs, const void *residual_in,
                                  const void *gamma, float eps, void *residual_out,
                                  void *const *y_out, double *inv_out, double *y64_out,
                                  int nthreads) {
    if (T < 0 || H <= 0 || N < 1 || !bufs || !residual_in || !residual_out || !gamma || !y_out)
        return -2;
    tp_job_t j = {dt, H, N, bufs, residual_in, residual_out, gamma, eps, y_out, inv_out, y64_out};
    int used = 0;
    for (int32_t r = 0; r < N; ++r) {
        int64_t r0, r1;
        oracle_tp_rows(T, N, r, &r0, &r1);
        /* run_rows numbers rows from 0: shift this rank's block there */
        tp_job_t jr = j;
        const int64_t off = r0 * H * elem_size(dt);
        const void *bq[64];
        void *yq[64];
        if (N > 64) return -2;
        for (int32_t q = 0; q < N; ++q) {
            bq[q] = (const char *)bufs[q] + off;
            yq[q] = (char *)y_out[q] + off;
        }
        jr.bufs = bq;
        jr.y_out = yq;
        jr.residual_in = (const char *)residual_in + off;
        jr.residual_out = (char *)residual_out + off;
        jr.inv_out = inv_out ? inv_out + r0 : NULL;
        jr.y64_out = y64_out ? y64_out + r0 * H : NULL;
        const int rc = run_rows(&jr, tp_row, r1 - r0, H, nthreads);
        if (rc < 0) return rc;
        if (rc > used) used = rc;
    }
    return used;
}

/* ----------------------------------------------------------------------- */
/* fp8 output                                                               */
/* ----------------------------------------------------------------------- */

/* The two 8-bit formats ("Block All Reduce", FP8 section: e4m3 and e5m2,
 * converted with saturation to the largest finite value):
 *   e4m3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; no infinity;
 *         S.1111.111 is NaN, so the largest finite value is 448 (S.1111.110);
 *   e5m2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits; IEEE-style
 *         infinities and NaNs; largest finite value 57344.
 * Both have gradual underflow (subnormal step 2^(emin - mbits)). */
typedef struct {
    int p, emin, emax, mbits, bias;
    double maxf;
} fp8_format;

static const fp8_format FP8[2] = {
    {4, -6, 8, 3, 7, 448.0},      /* e4m3 */
    {3, -14, 15, 2, 15, 57344.0}, /* e5m2 */
};

/* Round to nearest, ties to even, saturating: a value whose rounding would
 * exceed the largest finite value in magnitude gives +-maxf. */
static double round_fp8_sat(const fp8_format *f, double v) {
    if (isnan(v)) return v;
    double r = round_to_format(v, f->p, f->emin, f->emax);
    if (isinf(r) || fabs(r) > f->maxf) r = copysign(f->maxf, v);
    return r;
}

/* Code of a value that is exactly representable (finite or NaN). */
static uint8_t encode_fp8(const fp8_format *f, double v) {
    if (isnan(v)) return 0x7f;
    uint8_t s = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a == 0.0) return s;
    int e2;
    frexp(a, &e2);
    int lead = e2 - 1;
    if (lead >= f->emin) {
        int frac = (int)ldexp(a, f->mbits - lead) - (1 << f->mbits);
        return (uint8_t)(s | ((lead + f->bias) << f->mbits) | frac);
    }
    return (uint8_t)(s | (int)ldexp(a, f->mbits - f->emin)); /* subnormal */
}

static double decode_fp8(const fp8_format *f, uint8_t b) {
    int sign = b >> 7, e = (b & 0x7f) >> f->mbits, m = b & ((1 << f->mbits) - 1);
    int emax_field = (1 << (7 - f->mbits)) - 1;
    double v;
    if (e == 0)
        v = ldexp((double)m, f->emin - f->mbits);
    else if (f->mbits == 3 && e == emax_field && m == 7)
        v = NAN;
    else if (f->mbits == 2 && e == emax_field)
        v = m == 0 ? INFINITY : NAN;
    else
        v = ldexp((double)(m + (1 << f->mbits)), e - f->bias - f->mbits);
    return sign ? -v : v;
}

/*
 * The three operations with an 8-bit output.  h, inv and v_i = (h_i * inv) *
 * gamma_i as in one_row (binary64); then the code q_i = fp8(v_i / s):
 *   mode 0 (per tensor): s = the binary32 `scale` argument;
 *   mode 1 (per row):    s = max_i |v_i| / maxf (binary64; s = 1 for a row
 *                        of zeros), reported in row_scales_out[t] rounded to
 *                        binary32.
 * R = 0 plain, R >= 1 partials + residual (residual in the inputs' type,
 * updated in place).  codes: T rows of ldq bytes.  u64_out (optional, dense
 * [T, H]): v_i / s before the rounding.
 */
int oracle_rows_fp8(int dt, int fmt, int64_t T, int64_t H, int32_t R, const void *x, int64_t ldx,
                    int64_t slice, void *residual, int64_t ldr, const void *gamma, float eps,
                    int mode, float scale, uint8_t *codes, int64_t ldq, float *row_scales_out,
                    double *u64_out) {
    if (T < 0 || H <= 0 || ldx < H || ldq < H || (R >= 1 && (!residual || ldr < H)) ||
        (mode != 0 && mode != 1) || (fmt != 0 && fmt != 1) || !codes)
        return -2;
    const fp8_format *f = &FP8[fmt];
    double *h = (double *)malloc(sizeof(double) * (size_t)H);
    double *v = (double *)malloc(sizeof(double) * (size_t)H);
    if (!h || !v) {
        free(h);
        free(v);
        return -1;
    }
    for (int64_t t = 0; t < T; ++t) {
        /* h, inv: the same steps as one_row */
        const int64_t xrow = t * ldx, rrow = t * ldr;
        if (R == 0) {
            for (int64_t i = 0; i < H; ++i) h[i] = load_elem(dt, x, xrow + i);
        } else {
            for (int64_t i = 0; i < H; ++i) {
                float acc = (float)load_elem(dt, x, xrow + i);
                for (int32_t r = 1; r < R; ++r)
                    acc = acc + (float)load_elem(dt, x, (int64_t)r * slice + xrow + i);
                acc = acc + (float)load_elem(dt, residual, rrow + i);
                h[i] = round_dt(dt, (double)acc);
            }
            for (int64_t i = 0; i < H; ++i) store_exact(dt, residual, rrow + i, h[i]);
        }
        double ss = 0.0;
        for (int64_t i = 0; i < H; ++i) ss += h[i] * h[i];
        const double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
        double amax = 0.0;
        for (int64_t i = 0; i < H; ++i) {
            v[i] = (h[i] * inv) * load_elem(dt, gamma, i);
            if (fabs(v[i]) > amax) amax = fabs(v[i]);
        }
        double s = (double)scale;
        if (mode == 1) {
            s = amax > 0.0 ? amax / f->maxf : 1.0;
            if (row_scales_out) row_scales_out[t] = (float)s;
        }
        for (int64_t i = 0; i < H; ++i) {
            const double u = v[i] / s;
            if (u64_out) u64_out[t * H + i] = u;
            codes[t * ldq + i] = encode_fp8(f, round_fp8_sat(f, u));
        }
    }
    free(h);
    free(v);
    return 1;
}

/* Reduce + residual + RMSNorm over R partials of 8-bit codes (dense
 * [R, T, H]) with one binary32 scale per partial; residual [T, H] of type dt
 * updated in residual_out; y, gamma of type dt. */
typedef struct {
    int dt, fmt;
    int64_t T, H;
    int32_t R;
    const uint8_t *codes;
    const float *scales;
    const void *residual_in;
    const void *gamma;
    float eps;
    void *residual_out;
    void *y;
    double *inv_out;
    double *y64_out;
} fp8in_job_t;

static void fp8in_row(const void *ctx, int64_t t, double *h) {
    const fp8in_job_t *j = (const fp8in_job_t *)ctx;
    const fp8_format *f = &FP8[j->fmt];
    const int64_t H = j->H, row = t * H;
    for (int64_t i = 0; i < H; ++i) {
        /* each dequantised partial: one binary32 rounding of code * scale */
        float acc = (float)decode_fp8(f, j->codes[row + i]) * j->scales[0];
        for (int32_t r = 1; r < j->R; ++r) {
            const float v = (float)decode_fp8(f, j->codes[(int64_t)r * j->T * H + row + i]) *
                            j->scales[r];
            acc = acc + v;
        }
        acc = acc + (float)load_elem(j->dt, j->residual_in, row + i);
        h[i] = round_dt(j->dt, (double)acc);
    }
    if (j->residual_out)
        for (int64_t i = 0; i < H; ++i) store_exact(j->dt, j->residual_out, row + i, h[i]);
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) ss += h[i] * h[i];
    const double inv = 1.0 / sqrt(ss / (double)H + (double)j->eps);
    if (j->inv_out) j->inv_out[t] = inv;
    for (int64_t i = 0; i < H; ++i) {
        const double v = (h[i] * inv) * load_elem(j->dt, j->gamma, i);
        if (j->y64_out) j->y64_out[row + i] = v;
        store_exact(j->dt, j->y, row + i, round_dt(j->dt, v));
    }
}

int oracle_reduce_fp8in(int dt, int fmt, int64_t T, int64_t H, int32_t R, const uint8_t *codes,
                        const float *scales, const void *residual_in, const void *gamma, float eps,
                        void *residual_out, void *y, double *inv_out, double *y64_out,
                        int nthreads) {
    if (T < 0 || H <= 0 || R < 1 || (fmt != 0 && fmt != 1) || !codes || !scales ||
        !residual_in || !gamma || !y)
        return -2;
    fp8in_job_t j = {dt, fmt, T, H, R, codes, scales, residual_in, gamma, eps,
                     residual_out, y, inv_out, y64_out};
    return run_rows(&j, fp8in_row, T, H, nthreads);
}

int oracle_decode_fp8(int fmt, const uint8_t *src, double *dst, int64_t n) {
    if (fmt != 0 && fmt != 1) return -2;
    for (int64_t i = 0; i < n; ++i) dst[i] = decode_fp8(&FP8[fmt], src[i]);
    return 1;
}

int oracle_round_fp8(int fmt, const double *src, uint8_t *dst, int64_t n) {
    if (fmt != 0 && fmt != 1) return -2;
    for (int64_t i = 0; i < n; ++i) dst[i] = encode_fp8(&FP8[fmt], round_fp8_sat(&FP8[fmt], src[i]));
    return 1;
}

/* ----------------------------------------------------------------------- */
/* GEMM producer with the fused residual-add RMSNorm as its epilogue        */
/* ----------------------------------------------------------------------- */

/*
 * The partial that the fused form adds to the residual is produced by a
 * matrix product: P = A W^T, A [T, K] (activations), W [H, K] (a linear
 * layer's weight, output features by input features).  Per row t:
 *
 *   0. P_ti = sum_k A_tk W_ik: every product is exact in binary64 (at most
 *      48 significant bits), summed with Neumaier's compensated summation,
 *      so P_ti is the exact sum to within one binary64 rounding;
 *   1. h_ti = RN_dt(P_ti + r_ti): the epilogue adds the residual to the
 *      accumulator and rounds once to the storage type (the partial is
 *      never rounded on its own); residual <- h;
 *   2-4. as in one_row: ss, inv = 1 / sqrt(ss / H + eps), y = RN_dt((h inv) gamma).
 *
 * ("Tokenweave fused-RMSNorm-AR kernel", Code walkthrough, for steps 1-4;
 * "sm80 GEMM + ReduceScatter", the flux epilogue: the GEMM's epilogue
 * consumes the accumulator tile before anything is written.)
 *
 * Also reported per element: P (p64_out) and S = sum_k |A_tk W_ik|
 * (abs64_out), the scale of the rounding error any binary32 accumulation of
 * the same products can make.
 */
typedef struct {
    int dt;
    int64_t T, H, K;
    const void *A;
    int64_t lda;
    const double *W64; /* W decoded, [H, K] dense */
    void *residual;    /* [T] rows of ldr, type dt, updated in place */
    int64_t ldr;
    const void *gamma;
    float eps;
    void *y;
    int64_t ldy;
    double *p64_out, *abs64_out, *inv_out;
} gemm_job_t;

static void gemm_row(const void *ctx, int64_t t, double *scratch) {
    const gemm_job_t *g = (const gemm_job_t *)ctx;
    const int64_t H = g->H, K = g->K;
    double *h = scratch, *arow = scratch + H;
    for (int64_t k = 0; k < K; ++k) arow[k] = load_elem(g->dt, g->A, t * g->lda + k);
    for (int64_t i = 0; i < H; ++i) {
        const double *wrow = g->W64 + i * K;
        double s = 0.0, c = 0.0, a = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double prod = arow[k] * wrow[k];
            const double u = s + prod;
            c += fabs(s) >= fabs(prod) ? (s - u) + prod : (prod - u) + s;
            s = u;
            a += fabs(prod);
        }
        const double P = s + c;
        if (g->p64_out) g->p64_out[t * H + i] = P;
        if (g->abs64_out) g->abs64_out[t * H + i] = a;
        h[i] = round_dt(g->dt, P + load_elem(g->dt, g->residual, t * g->ldr + i));
    }
    for (int64_t i = 0; i < H; ++i) store_exact(g->dt, g->residual, t * g->ldr + i, h[i]);
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) ss += h[i] * h[i];
    const double inv = 1.0 / sqrt(ss / (double)H + (double)g->eps);
    if (g->inv_out) g->inv_out[t] = inv;
    for (int64_t i = 0; i < H; ++i)
        store_exact(g->dt, g->y, t * g->ldy + i,
                    round_dt(g->dt, (h[i] * inv) * load_elem(g->dt, g->gamma, i)));
}

int oracle_gemm_add_rms_norm(int dt, int64_t T, int64_t H, int64_t K, const void *A, int64_t lda,
                             const void *W, int64_t ldw, void *residual, int64_t ldr,
                             const void *gamma, float eps, void *y, int64_t ldy, double *p64_out,
                             double *abs64_out, double *inv_out, int nthreads) {
    if (T < 0 || H <= 0 || K <= 0 || lda < K || ldw < K || ldr < H || ldy < H || !A || !W ||
        !residual || !gamma || !y)
        return -2;
    double *W64 = (double *)malloc(sizeof(double) * (size_t)(H * K));
    if (!W64) return -1;
    for (int64_t i = 0; i < H; ++i)
        for (int64_t k = 0; k < K; ++k) W64[i * K + k] = load_elem(dt, W, i * ldw + k);
    gemm_job_t g = {dt, T, H, K, A, lda, W64, residual, ldr, gamma, eps, y, ldy,
                    p64_out, abs64_out, inv_out};
    const int rc = run_rows(&g, gemm_row, T, H + K, nthreads);
    free(W64);
    return rc;
}

/* Elementwise helpers exposed so the tests can pin the format code alone. */
void oracle_decode(int dt, const void *src, double *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(dt, src, i);
}

void oracle_round(int dt, const double *src, void *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) store_exact(dt, dst, i, round_dt(dt, src[i]));
}

int oracle_elem_size(int dt) { return elem_size(dt); }
