/*
 * linrec_oracle.c -- plain CPU oracle for the first-order linear-recurrence scan.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py load this library.  The CUDA
 * library under linear_recurrence_scan_fp32_gb300/csrc shares no code,
 * header, helper or constant with it, and neither includes the other.
 *
 * What it computes.  The POPCORNBENCH trace "Kimi-K2.6 l1_p9" (problem
 * statement; the same statement opens "FW-GLM-5-1 l1_p9") defines, for
 * tensors a, b of shape (B, L, D), each channel (batch index i, channel d)
 * independently:
 *
 *     h[i,0,d] = b[i,0,d]
 *     h[i,t,d] = a[i,t,d] * h[i,t-1,d] + b[i,t,d]      for 0 < t < L
 *
 * with a, b, h row-major and D contiguous: element (i,t,d) sits at offset
 * i*L*D + t*D + d.  A parallel scan reaches the same values (up to rounding
 * order) by associativity of the affine-map composition, so the oracle is the
 * definition itself: one sequential loop in t per channel.  a[i,0,d] is never
 * read (h_0 is b_0 by definition).
 *
 * Functions:
 *   linrec_oracle_f64     -- the definition in double precision (inputs
 *                            widened exactly from fp32), double output.
 *   linrec_oracle_f32seq  -- the same loop in fp32, one multiply and one add
 *                            per step, each rounded (the pages' PyTorch loop
 *                            `h = a[:, t] * h + b[:, t]` computes this).
 *   linrec_oracle_f64_channel -- one channel's whole sequence, for sampled
 *                            checks on workloads too large to hold in fp64.
 *   linrec_oracle_f64_carry -- the recurrence continued from a given state:
 *                            h[i,t,d] = a[i,t,d] * h[i,t-1,d] + b[i,t,d] for
 *                            every t >= 0, with h[i,-1,d] = h0[i,d] (so a_0
 *                            is used), and optionally the last state
 *                            h[i,L-1,d] written to hlast[i,d].  h0 = NULL
 *                            means the plain definition above.  This is the
 *                            running-h carry of "Kimi-K2.6 l1_p9" (the value
 *                            passed from one chunk to the next) exposed as an
 *                            argument, so a sequence can be scanned in segments.
 *   linrec_oracle_f64_backward -- the gradient of that recurrence for a loss
 *                            with dL/dh = g: with c_t = dL/dh_t in total,
 *                              c_{L-1} = g_{L-1} + dh_last,
 *                              c_t     = g_t + a_{t+1} * c_{t+1}      (t < L-1),
 *                              db_t = c_t,  da_t = c_t * h_{t-1},  dh0 = a_0 * c_0,
 *                            h_{-1} = h0 (or 0 without h0, when a_0 is unused
 *                            and da_0 = 0).  h is the forward output as given.
 *                            Not on the pages: it follows from the definition
 *                            by the chain rule.
 *   linrec_oracle_f64_bdl -- the same definition, carried from h0 like
 *                            linrec_oracle_f64_carry, for tensors laid out
 *                            (B, D, L) with time innermost: element (i, d, t)
 *                            at i*D*L + d*L + t, so each channel's sequence is
 *                            one contiguous row.  "Kimi-K2.6 l1_p9" weighs this
 *                            layout (its transpose discussion) as the one in
 *                            which a warp reads a channel's steps contiguously.
 *   linrec_oracle_decode16 / linrec_oracle_encode16 -- the two 16-bit storage
 *                            formats (kind 0: bfloat16, sign 1 / exponent 8 /
 *                            fraction 7 bits, bias 127; kind 1: IEEE 754
 *                            binary16, sign 1 / exponent 5 / fraction 10 bits,
 *                            bias 15).  decode16 gives a word's exact value from
 *                            its fields; encode16 rounds a double to the nearest
 *                            word, ties to the even significand, overflow to
 *                            infinity.  Not on the pages: they store the scan in
 *                            fp32 only.  A scan stored in 16 bits is, here, the
 *                            definition above applied to the decoded inputs, its
 *                            exact result then rounded once by encode16.
 *
 * Threads only split the set of independent channels; every channel is still
 * one sequential loop, so results do not depend on the thread count.
 * Compiled with -O2 -ffp-contract=off (no fused multiply-add, no fast-math).
 *
 * Parity pins (all in tests/test_oracle_pins.py): closed forms for a=1
 * (prefix sum), a=0 (copy), b=delta_0 (running product) and constant a, b
 * (geometric series); exact rational brute force of the expanded sum on tiny
 * inputs; the page's symbolic walk-through for t = 0, 1, 2; planted mistakes
 * that each pin must catch.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

typedef struct {
    const float *a, *b;
    void *h;
    int64_t B, L, D;
    int64_t n_units, d_per_unit, units_per_batch;
    int tid, nthreads;
    int f64;
} job_t;

/* One unit of work: batch index i, channels [d0, d1), all t. */
static void run_unit_f64(const float *a, const float *b, double *h,
                         int64_t L, int64_t D, int64_t i, int64_t d0, int64_t d1)
{
    const int64_t base = i * L * D;
    for (int64_t d = d0; d < d1; ++d)
        h[base + d] = (double)b[base + d];                 /* h_0 = b_0 */
    for (int64_t t = 1; t < L; ++t) {
        const int64_t row = base + t * D, prev = base + (t - 1) * D;
        for (int64_t d = d0; d < d1; ++d)
            h[row + d] = (double)a[row + d] * h[prev + d] + (double)b[row + d];
    }
}

static void run_unit_f32(const float *a, const float *b, float *h,
                         int64_t L, int64_t D, int64_t i, int64_t d0, int64_t d1)
{
    const int64_t base = i * L * D;
    for (int64_t d = d0; d < d1; ++d)
        h[base + d] = b[base + d];
    for (int64_t t = 1; t < L; ++t) {
        const int64_t row = base + t * D, prev = base + (t - 1) * D;
        for (int64_t d = d0; d < d1; ++d) {
            float prod = a[row + d] * h[prev + d];          /* rounded to fp32 */
            h[row + d] = prod + b[row + d];                 /* rounded to fp32 */
        }
    }
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    for (int64_t u = j->tid; u < j->n_units; u += j->nthreads) {
        int64_t i = u / j->units_per_batch;
        int64_t d0 = (u % j->units_per_batch) * j->d_per_unit;
        int64_t d1 = d0 + j->d_per_unit;
        if (d1 > j->D) d1 = j->D;
        if (d0 >= d1) continue;
        if (j->f64) run_unit_f64(j->a, j->b, (double *)j->h, j->L, j->D, i, d0, d1);
        else        run_unit_f32(j->a, j->b, (float *)j->h, j->L, j->D, i, d0, d1);
    }
    return NULL;
}

int linrec_oracle_hardware_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Returns the number of threads used (>= 1), or -1 on bad arguments. */
static int run(const float *a, const float *b, void *h, int64_t B, int64_t L, int64_t D,
               int nthreads, int f64)
{
    if (B < 0 || L < 0 || D < 0) return -1;
    if (B == 0 || L == 0 || D == 0) return 1;
    if (!a || !b || !h) return -1;
    if (nthreads <= 0) nthreads = linrec_oracle_hardware_threads();
    if (nthreads > 256) nthreads = 256;

    /* Split each batch's D channels into enough ranges to give every thread work. */
    int64_t ranges = (nthreads + B - 1) / B;
    if (ranges < 1) ranges = 1;
    if (ranges > D) ranges = D;
    int64_t d_per_unit = (D + ranges - 1) / ranges;
    int64_t units_per_batch = (D + d_per_unit - 1) / d_per_unit;
    int64_t n_units = B * units_per_batch;
    if ((int64_t)nthreads > n_units) nthreads = (int)n_units;

    job_t jobs[256];
    pthread_t th[256];
    for (int k = 0; k < nthreads; ++k) {
        jobs[k] = (job_t){a, b, h, B, L, D, n_units, d_per_unit, units_per_batch, k, nthreads, f64};
    }
    int started = 0;
    for (int k = 1; k < nthreads; ++k) {
        if (pthread_create(&th[k], NULL, worker, &jobs[k]) != 0) break;
        started = k;
    }
    /* Threads that failed to start: do their share here, in order. */
    for (int k = started + 1; k < nthreads; ++k) worker(&jobs[k]);
    worker(&jobs[0]);
    for (int k = 1; k <= started; ++k) pthread_join(th[k], NULL);
    return nthreads;
}

int linrec_oracle_f64(const float *a, const float *b, double *h,
                      int64_t B, int64_t L, int64_t D, int nthreads)
{
    return run(a, b, h, B, L, D, nthreads, 1);
}

int linrec_oracle_f32seq(const float *a, const float *b, float *h,
                         int64_t B, int64_t L, int64_t D, int nthreads)
{
    return run(a, b, h, B, L, D, nthreads, 0);
}

/* h_col[t] for t < L: the fp64 definition on channel (i, d) alone. */
int linrec_oracle_f64_channel(const float *a, const float *b, double *h_col,
                              int64_t B, int64_t L, int64_t D, int64_t i, int64_t d)
{
    if (B < 0 || L < 0 || D < 0 || i < 0 || i >= B || d < 0 || d >= D) return -1;
    if (L == 0) return 0;
    if (!a || !b || !h_col) return -1;
    const int64_t base = i * L * D + d;
    double h = (double)b[base];
    h_col[0] = h;
    for (int64_t t = 1; t < L; ++t) {
        const int64_t k = base + t * D;
        h = (double)a[k] * h + (double)b[k];
        h_col[t] = h;
    }
    return 0;
}

/* The recurrence continued from h0 (B x D, may be NULL), last state to hlast
   (B x D, may be NULL).  Sequential in t per channel, fp64 accumulator. */
int linrec_oracle_f64_carry(const float *a, const float *b, const double *h0, double *h, double *hlast,
                            int64_t B, int64_t L, int64_t D)
{
    if (B < 0 || L < 0 || D < 0) return -1;
    if (B == 0 || D == 0) return 0;
    if (!a || !b || (L > 0 && !h)) return -1;
    for (int64_t i = 0; i < B; ++i) {
        const int64_t base = i * L * D;
        for (int64_t d = 0; d < D; ++d) {
            double hv;
            int64_t t0;
            if (h0) {
                hv = h0[i * D + d];
                t0 = 0;
            } else {
                if (L == 0) { if (hlast) hlast[i * D + d] = 0.0; continue; }
                hv = (double)b[base + d];                       /* h_0 = b_0 */
                h[base + d] = hv;
                t0 = 1;
            }
            for (int64_t t = t0; t < L; ++t) {
                const int64_t k = base + t * D + d;
                hv = (double)a[k] * hv + (double)b[k];
                h[k] = hv;
            }
            if (hlast) hlast[i * D + d] = hv;
        }
    }
    return 0;
}

/* Gradient of the carried recurrence.  a, h, g: (B, L, D); h0, dhlast: (B, D) or NULL;
   da (may be NULL), db: (B, L, D) out; dh0: (B, D) out or NULL.  One reverse loop per channel. */
int linrec_oracle_f64_backward(const float *a, const float *h, const float *g, const double *h0,
                               const double *dhlast, double *da, double *db, double *dh0,
                               int64_t B, int64_t L, int64_t D)
{
    if (B < 0 || L < 0 || D < 0) return -1;
    if (B == 0 || D == 0 || L == 0) return 0;
    if (!a || !g || !db || (da && !h)) return -1;
    for (int64_t i = 0; i < B; ++i) {
        const int64_t base = i * L * D;
        for (int64_t d = 0; d < D; ++d) {
            double c = dhlast ? dhlast[i * D + d] : 0.0;    /* c_L: what flows in from after L-1 */
            double coef = 1.0;                              /* its weight in c_{L-1} */
            for (int64_t t = L - 1; t >= 0; --t) {
                const int64_t k = base + t * D + d;
                c = (double)g[k] + coef * c;                /* c_t = g_t + a_{t+1} c_{t+1} */
                db[k] = c;
                if (da) {
                    double hprev;
                    if (t > 0) hprev = (double)h[k - D];
                    else hprev = h0 ? h0[i * D + d] : 0.0;
                    da[k] = c * hprev;
                }
                coef = (double)a[k];                        /* a_t weighs c_t in c_{t-1} */
            }
            if (dh0) dh0[i * D + d] = coef * c;             /* a_0 * c_0 */
        }
    }
    return 0;
}

/* ---- 16-bit storage formats --------------------------------------------------
   A word is sign | exponent (ebits) | fraction (fbits).  Exponent field 0 holds
   zero and the subnormals 0.f x 2^(1-bias); the all-ones field holds infinity
   (fraction 0) and NaN; any other field e holds 1.f x 2^(e-bias). */
typedef struct { int ebits, fbits, bias; } fmt16_t;
static const fmt16_t kFmt16[2] = {{8, 7, 127}, {5, 10, 15}};   /* bfloat16, binary16 */

static double decode16(fmt16_t f, uint16_t w)
{
    const int emask = (1 << f.ebits) - 1;
    const int e = (w >> f.fbits) & emask;
    const int m = w & ((1 << f.fbits) - 1);
    double v;
    if (e == emask) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, 1 - f.bias - f.fbits);                 /* 0.f x 2^(1-bias) */
    else v = ldexp((double)((1 << f.fbits) | m), e - f.bias - f.fbits);         /* 1.f x 2^(e-bias) */
    return (w & 0x8000u) ? -v : v;
}

static uint16_t encode16(fmt16_t f, double x)
{
    const int emask = (1 << f.ebits) - 1;
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | (emask << f.fbits) | (1 << (f.fbits - 1)));   /* a quiet NaN */
    const double ax = fabs(x);
    if (isinf(ax)) return (uint16_t)(sign | (emask << f.fbits));
    if (ax == 0.0) return sign;
    int k = 0;
    frexp(ax, &k);                            /* 2^(k-1) <= ax < 2^k */
    int e = k - 1;                            /* ax's binade */
    const int emin = 1 - f.bias;              /* the smallest normal binade; below it the step stays */
    if (e < emin) e = emin;
    /* ax in steps of 2^(e - fbits), the spacing of the words in binade e: a power-of-two
       scaling, exact in double; rint rounds to the nearest step, ties to even */
    long long n = (long long)rint(ldexp(ax, f.fbits - e));
    if (n == (1ll << (f.fbits + 1))) {        /* rounded up into the next binade */
        n >>= 1;
        ++e;
    }
    if (n < (1ll << f.fbits))                 /* subnormal (e == emin): exponent field 0 */
        return (uint16_t)(sign | n);
    const int field = e + f.bias;
    if (field >= emask) return (uint16_t)(sign | (emask << f.fbits));   /* overflow: infinity */
    return (uint16_t)(sign | (field << f.fbits) | (n & ((1 << f.fbits) - 1)));
}

/* kind 0 = bfloat16, 1 = binary16.  Returns 0, or -1 on bad arguments. */
int linrec_oracle_decode16(int kind, const uint16_t *w, double *x, int64_t n)
{
    if (kind < 0 || kind > 1 || n < 0 || (n > 0 && (!w || !x))) return -1;
    for (int64_t i = 0; i < n; ++i) x[i] = decode16(kFmt16[kind], w[i]);
    return 0;
}

int linrec_oracle_encode16(int kind, const double *x, uint16_t *w, int64_t n)
{
    if (kind < 0 || kind > 1 || n < 0 || (n > 0 && (!w || !x))) return -1;
    for (int64_t i = 0; i < n; ++i) w[i] = encode16(kFmt16[kind], x[i]);
    return 0;
}

/* (B, D, L) layout: row i*D + d holds channel (i, d) over t = 0 .. L-1.
   h0, hlast: (B, D) or NULL, as in linrec_oracle_f64_carry. */
int linrec_oracle_f64_bdl(const float *a, const float *b, const double *h0, double *h, double *hlast,
                          int64_t B, int64_t D, int64_t L)
{
    if (B < 0 || L < 0 || D < 0) return -1;
    if (B == 0 || D == 0 || L == 0) return 0;
    if (!a || !b || !h) return -1;
    for (int64_t row = 0; row < B * D; ++row) {
        const float *ar = a + row * L;
        const float *br = b + row * L;
        double *hr = h + row * L;
        double hv = (double)br[0];                          /* h_0 = b_0 */
        if (h0) hv = (double)ar[0] * h0[row] + (double)br[0];   /* h_{-1} = h0: a_0 used */
        hr[0] = hv;
        for (int64_t t = 1; t < L; ++t) {
            hv = (double)ar[t] * hv + (double)br[t];
            hr[t] = hv;
        }
        if (hlast) hlast[row] = hv;
    }
    return 0;
}
