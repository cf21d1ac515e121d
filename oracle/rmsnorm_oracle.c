/*
 * rmsnorm_oracle.c -- plain, slow, obviously correct CPU reference for the RMSNorm
 * forward, the fused dX+dW backward and the fused residual-add + RMSNorm + E4M3 1x128
 * block quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference legs do.  It shares no code, header, table or constant with the CUDA path.
 *
 * Arithmetic: every floating-point step is IEEE binary64 unless a step is stated to be
 * binary32 (the block-quant part, whose decisions are defined in fp32).  Inputs are
 * decoded exactly from their storage format (fp32, bf16 or fp64) to binary64.  No
 * blocking, fusion or reordering beyond the definitions below.  Compile without
 * -ffast-math and with -ffp-contract=off so that no multiply-add is fused.
 *
 * Sources (page title, section):
 *  [CAKE]  FlashInfer PR #5741 "cake_rmsnorm_train: BF16 RMSNorm training forward +
 *          one-launch backward", sections Design (Forward, Backward), API, Accuracy,
 *          Determinism.
 *  [FQ]    FlashInfer PR #4480 "Add FusedAddRMSNormFP8BlockQuant", sections Summary,
 *          Kernel, API, and the review commit on the block-scale tolerance
 *          ("scale = amax/448").
 *  [MILES] miles-ext-kernels PR #15 (re-vendoring the Cake RMSNorm packages), section
 *          Accuracy (dW budget: atol 1e-4 + rtol 1e-4 of an FP64 sum at the forward's
 *          rstd).
 *  [OCP]   OCP 8-bit floating point specification, E4M3 encoding (bias 7, no
 *          infinities, S.1111.111 = NaN, largest finite 448).
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "binary32 steps must be evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

/* storage formats of the inputs */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

/* ------------------------------------------------------------------ decoding */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an IEEE binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* exact value of element i of a buffer stored in format dt */
static double elem(const void* p, int dt, int64_t i)
{
    if (dt == OR_F32) return (double)((const float*)p)[i];
    if (dt == OR_BF16) return bf16_bits_to_double(((const uint16_t*)p)[i]);
    return ((const double*)p)[i];
}

/* ------------------------------------------------------------------ rounding helpers */

/* Round a binary64 value to the nearest bfloat16 (8 significant bits, binary32
 * exponent range, subnormals kept), ties to even; results beyond the largest finite
 * bf16 round to infinity as IEEE round-to-nearest prescribes.  Returns the bit pattern. */
uint16_t or_bf16_round(double d)
{
    float f;
    uint32_t u;
    if (isnan(d)) return 0x7FC0;
    double a = fabs(d);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);                     /* a = m * 2^e with m in [0.5, 1) */
        int lead = e - 1;                 /* floor(log2 a) */
        if (lead < -126) lead = -126;     /* bf16 subnormal range: fixed quantum */
        double quantum = ldexp(1.0, lead - 7);
        double k = nearbyint(a / quantum); /* default rounding mode: ties to even */
        r = k * quantum;
        /* overflow threshold of round-to-nearest: (2 - 2^-8) * 2^127 and above -> inf */
        if (r >= ldexp(1.0, 128)) r = INFINITY;
    }
    f = (float)r; /* exact: r is representable in binary32 */
    memcpy(&u, &f, sizeof u);
    uint16_t bits = (uint16_t)(u >> 16);
    if (signbit(d)) bits |= 0x8000;
    return bits;
}

/* or_bf16_round over an array */
void or_bf16_round_n(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_round(v[i]);
}

/* OCP E4M3 ("FN") decode of one code, exact in binary32 */
float or_e4m3_decode(uint8_t code)
{
    int s = code >> 7, E = (code >> 3) & 0xF, M = code & 0x7;
    float v;
    if (E == 0xF && M == 0x7) return NAN;
    if (E == 0) v = ldexpf((float)M, -9);               /* subnormal: M/8 * 2^-6 */
    else v = ldexpf((float)(8 + M), E - 7 - 3);          /* (1 + M/8) * 2^(E-7) */
    return s ? -v : v;
}

/* OCP E4M3 encode of a binary32 value: round to nearest, ties to even; finite values
 * beyond +-448 (and infinities) saturate to +-448; NaN -> 0x7F.  The sign of zero is
 * kept (-0 -> 0x80). */
uint8_t or_e4m3_encode(float v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int lead = e - 1;                   /* floor(log2 a) */
    if (lead < -6) lead = -6;           /* subnormals share the quantum 2^-9 */
    double quantum = ldexp(1.0, lead - 3);
    double k = nearbyint(a / quantum);  /* exact division by a power of two; ties to even */
    double r = k * quantum;             /* rounded magnitude, <= 448 since a < 448 */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) {           /* subnormal code */
        return sign | (uint8_t)(int)(r / ldexp(1.0, -9));
    }
    frexp(r, &e);
    int E = (e - 1) + 7;
    int M = (int)(r / ldexp(1.0, e - 1 - 3)) - 8;
    return sign | (uint8_t)((E << 3) | M);
}

/* ------------------------------------------------------------------ threading */

typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);

typedef struct {
    range_fn fn;
    void* ctx;
    int64_t begin, end;
} job_t;

static void* run_job(void* arg)
{
    job_t* j = (job_t*)arg;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

/* Split [0, n) into nthreads contiguous pieces.  Every output element is computed by
 * exactly one piece with the same arithmetic whatever the split, so the results do not
 * depend on the thread count. */
static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    job_t jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].begin = n * t / nthreads;
        jobs[t].end = n * (t + 1) / nthreads;
        pthread_create(&th[t], NULL, run_job, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ forward */

typedef struct {
    const void* x; int x_dt;
    const void* w; int w_dt;
    int64_t H; double eps;
    double* y; double* rstd;
} fwd_ctx;

/* [CAKE] Design/Forward: per row, the mean of squares, rstd = 1/sqrt(mean + eps) and
 * y = x * rstd * w.  Here all of it in binary64 on the exact input values; y is the
 * unrounded value (the caller compares it with a rounded device output). */
static void fwd_rows(void* vctx, int64_t r0, int64_t r1)
{
    fwd_ctx* c = (fwd_ctx*)vctx;
    const int64_t H = c->H;
    for (int64_t i = r0; i < r1; ++i) {
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double v = elem(c->x, c->x_dt, i * H + j);
            ss += v * v;
        }
        double ms = ss / (double)H;
        double r = 1.0 / sqrt(ms + c->eps);
        c->rstd[i] = r;
        if (c->y) {
            for (int64_t j = 0; j < H; ++j)
                c->y[i * H + j] = elem(c->x, c->x_dt, i * H + j) * r * elem(c->w, c->w_dt, j);
        }
    }
}

/* x: [T, H] row-major in format x_dt; w: [H] in format w_dt.
 * Outputs (binary64): y [T, H] (may be NULL), rstd [T]. */
void or_rmsnorm_fwd(const void* x, int x_dt, const void* w, int w_dt, int64_t T, int64_t H,
                    double eps, double* y, double* rstd, int nthreads)
{
    fwd_ctx c = {x, x_dt, w, w_dt, H, eps, y, rstd};
    parallel_for(T, nthreads, fwd_rows, &c);
}

/* ------------------------------------------------------------------ backward */

typedef struct {
    const void* dy; const void* x; int x_dt;
    const void* w; int w_dt;
    const double* rstd;
    int64_t T, H;
    double* dx; double* dw;
} bwd_ctx;

/* [CAKE] Design/Backward: with xhat = x * rstd and g = dy * w,
 *   dx = rstd * (g - xhat * mean_j(g * xhat)).
 * rstd is an input (the forward's saved value), as the backward of the pages reads it. */
static void bwd_dx_rows(void* vctx, int64_t r0, int64_t r1)
{
    bwd_ctx* c = (bwd_ctx*)vctx;
    const int64_t H = c->H;
    for (int64_t i = r0; i < r1; ++i) {
        const double r = c->rstd[i];
        double dot = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double xh = elem(c->x, c->x_dt, i * H + j) * r;
            double g = elem(c->dy, c->x_dt, i * H + j) * elem(c->w, c->w_dt, j);
            dot += g * xh;
        }
        double mean = dot / (double)H;
        for (int64_t j = 0; j < H; ++j) {
            double xh = elem(c->x, c->x_dt, i * H + j) * r;
            double g = elem(c->dy, c->x_dt, i * H + j) * elem(c->w, c->w_dt, j);
            c->dx[i * H + j] = r * (g - xh * mean);
        }
    }
}

/* dW_j = sum over all rows i of dy_ij * x_ij * rstd_i  ([CAKE] Design/Backward; the
 * budget of [MILES] Accuracy is measured against exactly this FP64 sum).  Each column
 * is summed over the rows in row order with Neumaier's compensated summation; for bf16
 * x and dy with an fp32 rstd each term is exact in binary64 (8 + 8 + 24 significant
 * bits), so the column sum is within about one unit in the last place of the exact
 * sum.  Threads split the columns, so the result does not depend on the thread count. */
static void bwd_dw_cols(void* vctx, int64_t j0, int64_t j1)
{
    bwd_ctx* c = (bwd_ctx*)vctx;
    const int64_t H = c->H;
    const int64_t width = j1 - j0;
    if (width <= 0) return;
    double* s = (double*)calloc((size_t)width, sizeof(double));
    double* comp = (double*)calloc((size_t)width, sizeof(double));
    for (int64_t i = 0; i < c->T; ++i) {
        const double r = c->rstd[i];
        for (int64_t j = j0; j < j1; ++j) {
            double term = elem(c->dy, c->x_dt, i * H + j) * elem(c->x, c->x_dt, i * H + j) * r;
            double a = s[j - j0];
            double t = a + term;
            if (fabs(a) >= fabs(term)) comp[j - j0] += (a - t) + term;
            else comp[j - j0] += (term - t) + a;
            s[j - j0] = t;
        }
    }
    for (int64_t j = j0; j < j1; ++j) c->dw[j] = s[j - j0] + comp[j - j0];
    free(s);
    free(comp);
}

/* dy, x: [T, H] in format x_dt; w: [H] in w_dt; rstd: [T] binary64.
 * Outputs: dx [T, H] binary64 (may be NULL), dw [H] binary64 (may be NULL). */
void or_rmsnorm_bwd(const void* dy, const void* x, int x_dt, const void* w, int w_dt,
                    const double* rstd, int64_t T, int64_t H, double* dx, double* dw,
                    int nthreads)
{
    bwd_ctx c = {dy, x, x_dt, w, w_dt, rstd, T, H, dx, dw};
    if (dx) parallel_for(T, nthreads, bwd_dx_rows, &c);
    if (dw) parallel_for(H, nthreads, bwd_dw_cols, &c);
}

/* ------------------------------------------------------------------ fused add + norm */

typedef struct {
    const uint16_t* x; const uint16_t* res; const uint16_t* w;
    int64_t H; double eps;
    uint16_t* h_out; double* n_out; double* rstd;
} fused_ctx;

/* [FQ] Summary/Kernel and [CAKE] Design/Forward (residual form): h = bf16(x + residual)
 * is the value written back to the residual and the value that is normalized; the
 * normed output is h * rstd * w with rstd = 1/sqrt(mean(h^2) + eps).  The sum x + r of
 * two bf16 values is formed exactly in binary64 and rounded once to bf16. */
static void fused_rows(void* vctx, int64_t r0, int64_t r1)
{
    fused_ctx* c = (fused_ctx*)vctx;
    const int64_t H = c->H;
    for (int64_t i = r0; i < r1; ++i) {
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double sum = bf16_bits_to_double(c->x[i * H + j]) + bf16_bits_to_double(c->res[i * H + j]);
            uint16_t hb = or_bf16_round(sum);
            c->h_out[i * H + j] = hb;
            double h = bf16_bits_to_double(hb);
            ss += h * h;
        }
        double r = 1.0 / sqrt(ss / (double)H + c->eps);
        c->rstd[i] = r;
        for (int64_t j = 0; j < H; ++j)
            c->n_out[i * H + j] = bf16_bits_to_double(c->h_out[i * H + j]) * r * bf16_bits_to_double(c->w[j]);
    }
}

/* x, residual: [T, H] bf16 bits; w: [H] bf16 bits.
 * Outputs: h_out [T, H] bf16 bits (the updated residual), n_out [T, H] binary64
 * (unrounded normed value), rstd [T] binary64. */
void or_fused_add_rmsnorm(const uint16_t* x, const uint16_t* residual, const uint16_t* w,
                          int64_t T, int64_t H, double eps, uint16_t* h_out, double* n_out,
                          double* rstd, int nthreads)
{
    fused_ctx c = {x, residual, w, H, eps, h_out, n_out, rstd};
    parallel_for(T, nthreads, fused_rows, &c);
}

/* ------------------------------------------------------------------ 1x128 block quant */

typedef struct {
    const uint16_t* n; int64_t H; int64_t ld;
    uint8_t* q; float* scale;
} quant_ctx;

/* [FQ] Summary/Kernel/API: each row is split into blocks of 128 consecutive columns.
 * For block b of row m, in binary32 arithmetic:
 *   amax = max |n|                      (exact: a maximum of bf16 values)
 *   scale = amax / 448                  (448 = largest finite E4M3 value)
 *   q = E4M3(n / scale)                 (round to nearest even, saturating)
 * The scale of (row m, block b) is stored at scale[b * ld + m]: the (H/128, ld) buffer,
 * unit stride along the rows.  A block whose amax is 0 stores scale 0 and the signed
 * zero code of each element (no division is made). */
static void quant_rows(void* vctx, int64_t r0, int64_t r1)
{
    quant_ctx* c = (quant_ctx*)vctx;
    const int64_t H = c->H, nb = H / 128;
    for (int64_t m = r0; m < r1; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t* blk = c->n + m * H + b * 128;
            float amax = 0.0f;
            for (int k = 0; k < 128; ++k) {
                float a = fabsf((float)bf16_bits_to_double(blk[k]));
                if (a > amax) amax = a;
            }
            float scale = amax / 448.0f; /* binary32 division, correctly rounded */
            c->scale[b * c->ld + m] = scale;
            for (int k = 0; k < 128; ++k) {
                float v = (float)bf16_bits_to_double(blk[k]);
                float qv = (scale > 0.0f) ? v / scale : v;
                c->q[m * H + b * 128 + k] = or_e4m3_encode(qv);
            }
        }
    }
}

/* n: [T, H] bf16 bits (the normed values to quantize), H % 128 == 0.
 * Outputs: q [T, H] E4M3 codes; scale as described above with leading dimension ld.
 * Entries scale[b * ld + m] for m >= T are not written. */
void or_block_quant_e4m3(const uint16_t* n, int64_t T, int64_t H, uint8_t* q, float* scale,
                         int64_t ld, int nthreads)
{
    quant_ctx c = {n, H, ld, q, scale};
    parallel_for(T, nthreads, quant_rows, &c);
}
