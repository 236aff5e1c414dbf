/*
 * CPU oracle for the ternary-weight linear layer, its backward and AdamW.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, fp64 statement of
 * what the GPU library computes.  It shares no code, header, table or helper
 * with the CUDA path, and only the tests, the smoke check and the bench's CPU
 * baseline may load it.  Nothing in the library calls it.
 *
 * Sources (the page that defines each step):
 *   train_gpu.cu (on-device RWKV-x SR4 training driver)
 *     - header comment "Optimizer split": W_eff[r,c] = scale[c]*ternary(q)[r,c],
 *       q an int4 accumulator, per-OUTPUT-COLUMN scale; SR4_THETA = 2,
 *       SR4_Q_CLAMP = 7.
 *     - device glue kernels: tg_tern_from_q (w = sign(q) if |q| >= theta else 0),
 *       tg_apply_scale (row-major [rows, cols], c = column), tg_gq
 *       (gq = grad * scale[c]), tg_scale_grad (sgrad[c] = sum over r of
 *       grad[r,c] * tern[r,c], in double, r ascending).
 *     - resident optimizer launchers: adamw_dev (bias corrections 1 - beta^t,
 *       is_adamw flag), and the step loop that scales the scale gradient by
 *       scale_lr/lr before the scales' AdamW step.
 *   heal_gpu.rs (DTG-MA mask training): the host Adam update, which places eps
 *     outside the square root of the bias-corrected second moment.
 *
 * Conventions: X [M][K] and dY [M][N] are bf16 bit patterns (uint16), q [K][N]
 * int8, scale [N] fp32, every matrix row-major.  K = rows r = input features,
 * N = cols c = output features, M = tokens.  All sums are fp64 in ascending
 * index order.  "abs" outputs are the sums of |term| of each output's dot
 * product, the denominators of the comparison tolerance.
 *
 * SR4 q-update (or_sr4_*): PARITY UNPINNED.  The page names fc_sr4_scale and
 * fc_sr4_update but does not print their bodies; the functions below state the
 * plainest reading of their arguments and are pinned only by invariants.
 *
 * Readings where the pages leave a step open:
 *   - the AdamW body is not on the pages: decoupled decay uses the old weight,
 *     w' = w - lr*wd*w - lr*mhat/(sqrt(vhat)+eps); with decoupled = 0 the decay
 *     is folded into the gradient (g += wd*w), the plain Adam-with-L2 form;
 *   - gmul multiplies the gradient before the step (the page's scale_lr/lr);
 *   - bf16 rounding of a scale is round-to-nearest, ties to even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- scalars */

/* train_gpu.cu, tg_tern_from_q: +1 when q >= theta, -1 when q <= -theta, else 0. */
int or_ternary(int q, int theta) {
    if (q >= theta) return 1;
    if (q <= -theta) return -1;
    return 0;
}

/* Saturate the int8 accumulator to [-clamp, clamp] (SR4_Q_CLAMP = 7 on the page). */
int or_clamp(int q, int clamp) {
    if (q > clamp) return clamp;
    if (q < -clamp) return -clamp;
    return q;
}

/* A bf16 bit pattern is the upper half of an IEEE binary32: value = bits << 16. */
double or_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* bf16 (8 significant bits, binary32 exponent range) nearest to x, ties to
 * even, for finite normal-range x or zero; returned as its bit pattern. */
uint16_t or_bf16_round(double x) {
    if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
    int e;
    double m = frexp(fabs(x), &e);          /* |x| = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(ldexp(m, 8));      /* 8 significant bits, ties to even */
    double v = ldexp(r, e - 8);
    float f = (float)(x < 0 ? -v : v);      /* exact: v has 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* x rounded to a binary floating-point grid of p significant bits whose smallest
 * normal exponent is emin (below it the spacing stays 2^(emin-p+1): subnormals),
 * ties to even, with unbounded exponent range above.  The caller handles overflow. */
static double or_round_grid(double x, int p, int emin) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(fabs(x), &e);                     /* floor(log2|x|) = e - 1 */
    int lsb = (e - 1 > emin ? e - 1 : emin) - (p - 1);   /* exponent of one unit in the last place */
    double r = ldexp(nearbyint(ldexp(fabs(x), -lsb)), lsb);   /* default rounding: ties to even */
    return x < 0 ? -r : r;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 * normal values 2^-14 .. 65504, subnormals k * 2^-24.  Value of a bit pattern. */
double or_f16_value(uint16_t h) {
    int sgn = h >> 15, ex = (h >> 10) & 0x1F, fr = h & 0x3FF;
    double v;
    if (ex == 0x1F) v = fr ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)fr, -24);
    else v = ldexp(1.0 + fr / 1024.0, ex - 15);
    return sgn ? -v : v;
}

/* binary16 nearest to x, ties to even; beyond 65504 + half a unit it is infinity
 * (IEEE 754 round to nearest).  Finite x; returned as its bit pattern. */
uint16_t or_f16_round(double x) {
    uint16_t sgn = signbit(x) ? 0x8000u : 0u;
    double r = fabs(or_round_grid(x, 11, -14));
    if (r == 0.0) return sgn;
    if (r > 65504.0) return sgn | 0x7C00u;
    int e;
    frexp(r, &e);
    if (e - 1 < -14) return sgn | (uint16_t)ldexp(r, 24);   /* subnormal: r / 2^-24 */
    return sgn | (uint16_t)((e - 1 + 15) << 10) | (uint16_t)(ldexp(r, -(e - 1)) * 1024.0 - 1024.0);
}

/* 8-bit E4M3 (OCP 8-bit floating point, the tensor cores' e4m3): 1 sign bit, 4
 * exponent bits (bias 7), 3 fraction bits, no infinities, S.1111.111 = NaN;
 * normal values 2^-6 .. 448, subnormals k * 2^-9.  Value of a bit pattern. */
double or_e4m3_value(uint8_t b) {
    int sgn = b >> 7, ex = (b >> 3) & 0xF, fr = b & 7;
    double v;
    if (ex == 0xF && fr == 7) v = NAN;
    else if (ex == 0) v = ldexp((double)fr, -9);
    else v = ldexp(1.0 + fr / 8.0, ex - 7);
    return sgn ? -v : v;
}

/* E4M3 nearest to x, ties to even, saturating: a magnitude that rounds above 448
 * becomes 448 (the "satfinite" conversion).  Finite x; returned as its bit pattern. */
uint8_t or_e4m3_round(double x) {
    uint8_t sgn = signbit(x) ? 0x80u : 0u;
    double r = fabs(or_round_grid(x, 4, -6));
    if (r == 0.0) return sgn;
    if (r > 448.0) r = 448.0;
    int e;
    frexp(r, &e);
    if (e - 1 < -6) return sgn | (uint8_t)ldexp(r, 9);      /* subnormal: r / 2^-9 */
    return sgn | (uint8_t)((e - 1 + 7) << 3) | (uint8_t)(ldexp(r, -(e - 1)) * 8.0 - 8.0);
}

/* ------------------------------------------------------------ materialise */

/*
 * Clamp, ternarise and encode one weight matrix q [K][N].
 *   qc     [K][N]    clamped q (may be NULL)
 *   packed [K][N/16] 2-bit codes, element (r,c) in word r*(N/16) + c/16 at bits
 *                    2*(c%16): 0 -> 00, +1 -> 01, -1 -> 11 (may be NULL)
 *   t      [K][N]    bf16 of T (may be NULL)
 *   whi    [K][N]    bf16 of s_hi[c]*T, s_hi = bf16(scale[c]) (may be NULL)
 *   wlo    [K][N]    bf16 of s_lo[c]*T, s_lo = bf16(scale[c] - s_hi) (may be NULL)
 *                    (T = 0 gives +0 = 0x0000 in t, whi and wlo; T = -1 with
 *                    s_lo = +0 gives -0 = 0x8000, the IEEE product)
 * N must be a multiple of 16 when packed is requested.
 */
void or_materialize(const int8_t* q, const float* scale, int64_t K, int64_t N, int theta, int clamp,
                    int8_t* qc, uint32_t* packed, uint16_t* t, uint16_t* whi, uint16_t* wlo) {
    for (int64_t r = 0; r < K; ++r) {
        for (int64_t c = 0; c < N; ++c) {
            int64_t i = r * N + c;
            int v = or_clamp(q[i], clamp);
            int w = or_ternary(v, theta);
            if (qc) qc[i] = (int8_t)v;
            if (packed) {
                uint32_t code = w == 1 ? 1u : (w == -1 ? 3u : 0u);
                uint32_t* word = &packed[r * (N / 16) + c / 16];
                if (c % 16 == 0) *word = 0;
                *word |= code << (2 * (c % 16));
            }
            if (t) t[i] = or_bf16_round((double)w);
            if (whi || wlo) {
                double s = (double)scale[c];
                double shi = or_bf16_value(or_bf16_round(s));
                double slo = or_bf16_value(or_bf16_round(s - shi));
                /* a zero weight encodes as +0 in every plane */
                if (whi) whi[i] = w == 0 ? 0x0000u : or_bf16_round(shi * w);
                if (wlo) wlo[i] = w == 0 ? 0x0000u : or_bf16_round(slo * w);
            }
        }
    }
}

/*
 * The dX operands of the fp16 + e4m3 split (this library's encoding; the pages
 * form W_eff = scale[c]*T in fp32).  Per column, scale[c] = a_c * 2^e_c with
 * e_c = floor(log2|scale[c]|) and a_c in +-[1, 2) (a_c = 0, e_c = 0 for a zero
 * scale):
 *   wh16 [K][N] binary16 of h_c * T,           h_c = f16(a_c)
 *   wl8  [K][N] e4m3 of l_c * T,               l_c = e4m3(2^7 * (a_c - h_c))
 * so that h_c + 2^-7 * l_c = a_c within 2^-15 |a_c|.  A zero weight is +0 in both
 * planes; a negative one flips the sign bit (so l_c = +0 with T = -1 gives -0).
 */
void or_split8_planes(const int8_t* q, const float* scale, int64_t K, int64_t N, int theta, int clamp,
                      uint16_t* wh16, uint8_t* wl8) {
    for (int64_t c = 0; c < N; ++c) {
        double s = (double)scale[c], a = 0.0;
        if (s != 0.0) {
            int e;
            frexp(fabs(s), &e);
            a = ldexp(s, -(e - 1));                 /* exact: a power-of-two rescale */
        }
        uint16_t h = or_f16_round(a);
        uint8_t l = or_e4m3_round(ldexp(a - or_f16_value(h), 7));   /* a - h is exact in fp64 */
        for (int64_t r = 0; r < K; ++r) {
            int64_t i = r * N + c;
            int w = or_ternary(or_clamp(q[i], clamp), theta);
            if (wh16) wh16[i] = w == 0 ? 0x0000u : (uint16_t)(w < 0 ? h ^ 0x8000u : h);
            if (wl8) wl8[i] = w == 0 ? 0x00u : (uint8_t)(w < 0 ? l ^ 0x80u : l);
        }
    }
}

/* ------------------------------------------------------------ threading */

typedef struct {
    void (*fn)(void* ctx, int64_t lo, int64_t hi);
    void* ctx;
    int64_t lo, hi;
} or_part;

static void* or_part_run(void* a) {
    or_part* p = (or_part*)a;
    p->fn(p->ctx, p->lo, p->hi);
    return NULL;
}

/* Split [0, n) into contiguous ranges over nthreads; every output is computed
 * by exactly one thread in its own fixed order, so threads change no result. */
static void or_parallel(void (*fn)(void*, int64_t, int64_t), void* ctx, int64_t n, int nthreads) {
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads > 64) nthreads = 64;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads <= 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[64];
    int live[64];
    or_part parts[64];
    for (int t = 0; t < nthreads; ++t) {
        parts[t].fn = fn;
        parts[t].ctx = ctx;
        parts[t].lo = n * t / nthreads;
        parts[t].hi = n * (t + 1) / nthreads;
        live[t] = pthread_create(&th[t], NULL, or_part_run, &parts[t]) == 0;
        if (!live[t]) fn(ctx, parts[t].lo, parts[t].hi);
    }
    for (int t = 0; t < nthreads; ++t)
        if (live[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------ forward */

typedef struct {
    const uint16_t *X, *dY;
    const int8_t* q;
    const float* scale;
    int64_t M, K, N;
    int theta;
    double *out, *outabs, *out2, *out2abs;
} or_lin;

/* Y[m][c] = scale[c] * sum_r X[m][r] * T[r][c]   (train_gpu.cu header: Y = X * W_eff). */
static void or_fwd_rows(void* vctx, int64_t m0, int64_t m1) {
    const or_lin* a = (const or_lin*)vctx;
    double* acc = (double*)malloc(sizeof(double) * (size_t)a->N * 2);
    double* aab = acc + a->N;
    for (int64_t m = m0; m < m1; ++m) {
        for (int64_t c = 0; c < a->N; ++c) acc[c] = aab[c] = 0.0;
        for (int64_t r = 0; r < a->K; ++r) {
            double x = or_bf16_value(a->X[m * a->K + r]);
            const int8_t* qrow = a->q + r * a->N;
            for (int64_t c = 0; c < a->N; ++c) {
                double term = x * (double)or_ternary(qrow[c], a->theta);
                acc[c] += term;
                aab[c] += fabs(term);
            }
        }
        for (int64_t c = 0; c < a->N; ++c) {
            double s = (double)a->scale[c];
            a->out[m * a->N + c] = s * acc[c];
            if (a->outabs) a->outabs[m * a->N + c] = fabs(s) * aab[c];
        }
    }
    free(acc);
}

void or_fwd(const uint16_t* X, const int8_t* q, const float* scale, int64_t M, int64_t K, int64_t N,
            int theta, double* Y, double* Yabs, int nthreads) {
    or_lin a = {X, NULL, q, scale, M, K, N, theta, Y, Yabs, NULL, NULL};
    or_parallel(or_fwd_rows, &a, M, nthreads);
}

/* ------------------------------------------------------------ dX */

/* dX[m][r] = sum_c dY[m][c] * scale[c] * T[r][c]   (dX = dY * W_eff^T). */
static void or_dx_rows(void* vctx, int64_t m0, int64_t m1) {
    const or_lin* a = (const or_lin*)vctx;
    double* dy = (double*)malloc(sizeof(double) * (size_t)a->N);
    for (int64_t m = m0; m < m1; ++m) {
        for (int64_t c = 0; c < a->N; ++c) dy[c] = or_bf16_value(a->dY[m * a->N + c]);
        for (int64_t r = 0; r < a->K; ++r) {
            const int8_t* qrow = a->q + r * a->N;
            double s = 0.0, sa = 0.0;
            for (int64_t c = 0; c < a->N; ++c) {
                double term = dy[c] * (double)a->scale[c] * (double)or_ternary(qrow[c], a->theta);
                s += term;
                sa += fabs(term);
            }
            a->out[m * a->K + r] = s;
            if (a->outabs) a->outabs[m * a->K + r] = sa;
        }
    }
    free(dy);
}

void or_dx(const uint16_t* dY, const int8_t* q, const float* scale, int64_t M, int64_t K, int64_t N,
           int theta, double* dX, double* dXabs, int nthreads) {
    or_lin a = {NULL, dY, q, scale, M, K, N, theta, dX, dXabs, NULL, NULL};
    or_parallel(or_dx_rows, &a, M, nthreads);
}

/* ------------------------------------------------------------ dW, gq, sgrad */

/*
 * G[r][c] = sum_m X[m][r] * dY[m][c]            (dL/dW_eff, ascending m)
 * gq[r][c] = G[r][c] * scale[c]                  (train_gpu.cu, tg_gq)
 * gq's abs sum: sum_m |X[m][r] * dY[m][c]| * |scale[c]|
 * Rows r0..r1 of G; used for gq and, per column, for sgrad.
 */
static void or_g_rows(void* vctx, int64_t r0, int64_t r1) {
    const or_lin* a = (const or_lin*)vctx;
    /* out = G rows, outabs = sum |X dY| rows; rows indexed by r */
    for (int64_t r = r0; r < r1; ++r) {
        double* g = a->out + r * a->N;
        double* ga = a->outabs + r * a->N;
        for (int64_t c = 0; c < a->N; ++c) g[c] = ga[c] = 0.0;
        for (int64_t m = 0; m < a->M; ++m) {
            double x = or_bf16_value(a->X[m * a->K + r]);
            const uint16_t* dyrow = a->dY + m * a->N;
            for (int64_t c = 0; c < a->N; ++c) {
                double term = x * or_bf16_value(dyrow[c]);
                g[c] += term;
                ga[c] += fabs(term);
            }
        }
    }
}

/*
 * gq [K][N], sgrad [N] and their abs sums (any output pointer may be NULL).
 * sgrad[c] = sum_r G[r][c] * T[r][c], r ascending (train_gpu.cu, tg_scale_grad);
 * its abs sum is sum_r sum_m |X[m][r] * dY[m][c] * T[r][c]|.
 */
void or_dw(const uint16_t* X, const uint16_t* dY, const int8_t* q, const float* scale, int64_t M,
           int64_t K, int64_t N, int theta, double* gq, double* gqabs, double* sgrad, double* sgradabs,
           int nthreads) {
    double* G = (double*)malloc(sizeof(double) * (size_t)(K * N));
    double* Ga = (double*)malloc(sizeof(double) * (size_t)(K * N));
    or_lin a = {X, dY, q, scale, M, K, N, theta, G, Ga, NULL, NULL};
    or_parallel(or_g_rows, &a, K, nthreads);
    for (int64_t r = 0; r < K; ++r)
        for (int64_t c = 0; c < N; ++c) {
            double s = (double)scale[c];
            if (gq) gq[r * N + c] = G[r * N + c] * s;
            if (gqabs) gqabs[r * N + c] = Ga[r * N + c] * fabs(s);
        }
    for (int64_t c = 0; c < N; ++c) {
        double s = 0.0, sa = 0.0;
        for (int64_t r = 0; r < K; ++r) {
            int w = or_ternary(q[r * N + c], theta);
            s += G[r * N + c] * (double)w;
            sa += Ga[r * N + c] * (double)abs(w);
        }
        if (sgrad) sgrad[c] = s;
        if (sgradabs) sgradabs[c] = sa;
    }
    free(G);
    free(Ga);
}

/* ------------------------------------------------------------ sampled entries */

/*
 * Single entries of the same outputs, for layers too large to evaluate whole.
 * The row/column operands are passed in directly:
 *   or_fwd_at  : Y[m][c]   from xrow = X[m][:] (K), qcol = q[:][c] (K), s = scale[c]
 *   or_dx_at   : dX[m][r]  from dyrow = dY[m][:] (N), qrow = q[r][:] (N), scale (N)
 *   or_gq_at   : gq[r][c]  from xcol = X[:][r] (M), dycol = dY[:][c] (M), s = scale[c]
 *   or_sgrad_at: sgrad[c]  from X (M*K, whole), dycol = dY[:][c] (M), qcol = q[:][c] (K)
 */
void or_fwd_at(const uint16_t* xrow, const int8_t* qcol, float s, int64_t K, int theta, double* out,
               double* outabs) {
    double acc = 0.0, aab = 0.0;
    for (int64_t r = 0; r < K; ++r) {
        double term = or_bf16_value(xrow[r]) * (double)or_ternary(qcol[r], theta);
        acc += term;
        aab += fabs(term);
    }
    *out = (double)s * acc;
    *outabs = fabs((double)s) * aab;
}

void or_dx_at(const uint16_t* dyrow, const int8_t* qrow, const float* scale, int64_t N, int theta,
              double* out, double* outabs) {
    double acc = 0.0, aab = 0.0;
    for (int64_t c = 0; c < N; ++c) {
        double term = or_bf16_value(dyrow[c]) * (double)scale[c] * (double)or_ternary(qrow[c], theta);
        acc += term;
        aab += fabs(term);
    }
    *out = acc;
    *outabs = aab;
}

void or_gq_at(const uint16_t* xcol, const uint16_t* dycol, float s, int64_t M, double* out,
              double* outabs) {
    double acc = 0.0, aab = 0.0;
    for (int64_t m = 0; m < M; ++m) {
        double term = or_bf16_value(xcol[m]) * or_bf16_value(dycol[m]);
        acc += term;
        aab += fabs(term);
    }
    *out = acc * (double)s;
    *outabs = aab * fabs((double)s);
}

typedef struct {
    const uint16_t *X, *dycol;
    const int8_t* qcol;
    int64_t M, K;
    int theta;
    double *G, *Ga;
} or_scol;

static void or_scol_rows(void* vctx, int64_t r0, int64_t r1) {
    const or_scol* a = (const or_scol*)vctx;
    for (int64_t r = r0; r < r1; ++r) {
        double g = 0.0, ga = 0.0;
        for (int64_t m = 0; m < a->M; ++m) {
            double term = or_bf16_value(a->X[m * a->K + r]) * or_bf16_value(a->dycol[m]);
            g += term;
            ga += fabs(term);
        }
        a->G[r] = g;
        a->Ga[r] = ga;
    }
}

void or_sgrad_at(const uint16_t* X, const uint16_t* dycol, const int8_t* qcol, int64_t M, int64_t K,
                 int theta, double* out, double* outabs, int nthreads) {
    double* G = (double*)malloc(sizeof(double) * (size_t)K * 2);
    or_scol a = {X, dycol, qcol, M, K, theta, G, G + K};
    or_parallel(or_scol_rows, &a, K, nthreads);
    double s = 0.0, sa = 0.0;
    for (int64_t r = 0; r < K; ++r) {
        int w = or_ternary(qcol[r], theta);
        s += G[r] * (double)w;
        sa += G[K + r] * (double)abs(w);
    }
    *out = s;
    *outabs = sa;
    free(G);
}

/* ------------------------------------------------------------ AdamW */

/*
 * One AdamW step in fp64 on n elements (train_gpu.cu, adamw_dev / fc_adamw_update
 * call: bc_i = 1 - beta_i^t; heal_gpu.rs: eps outside the square root).
 *   g' = gmul*g  (+ wd*w when decoupled == 0)
 *   m' = b1*m + (1-b1)*g'
 *   v' = b2*v + (1-b2)*g'^2
 *   w' = w - [decoupled] lr*wd*w - lr * (m'/bc1) / (sqrt(v'/bc2) + eps)
 * The hyper-parameters are the caller's fp32 values, widened to double.
 */
void or_adamw(const float* w, const float* g, const float* m, const float* v, int64_t n, int t, double lr,
              double b1, double b2, double eps, double wd, double gmul, int decoupled, double* w_out,
              double* m_out, double* v_out) {
    double bc1 = 1.0 - pow(b1, (double)t);
    double bc2 = 1.0 - pow(b2, (double)t);
    for (int64_t i = 0; i < n; ++i) {
        double wi = (double)w[i];
        double gi = gmul * (double)g[i];
        if (!decoupled) gi += wd * wi;
        double mi = b1 * (double)m[i] + (1.0 - b1) * gi;
        double vi = b2 * (double)v[i] + (1.0 - b2) * gi * gi;
        double step = lr * (mi / bc1) / (sqrt(vi / bc2) + eps);
        double decay = decoupled ? lr * wd * wi : 0.0;
        w_out[i] = wi - decay - step;
        m_out[i] = mi;
        v_out[i] = vi;
    }
}

/* ------------------------------------------------------------ SR4 q-update */

/*
 * SR4 step on one ternary matrix's accumulator q (page "train_gpu.cu": sr4_dev
 * calls fc_sr4_scale<<<1,1>>>(gq, numel, inv_bs, target_step, d_s) and then
 * fc_sr4_update(q, gq, numel, inv_bs, d_s, seed, idx_base, counter, q_clamp,
 * use_dither); both bodies are off the page).  PARITY UNPINNED: the oracle
 * states the plainest reading of those names, and only invariants pin it:
 *
 *   step scalar   s = target_step / mean_i |gq_i * inv_bs|      (s = 0 when the mean is 0)
 *                 so that the mean requested step is target_step accumulator units;
 *   update        x_i = (gq_i * inv_bs) * s
 *                 q_i <- clamp(q_i - floor(x_i + u_i), -q_clamp, q_clamp)
 *                 with u_i ~ U[0,1) from the counter RNG (use_dither), else u_i = 1/2:
 *                 stochastic rounding of the descent step -x_i into the int4 accumulator
 *                 ("SR4"), E[q_new - q] = -x_i away from the clamp;
 *                 a non-finite x_i leaves q_i unchanged.
 *
 * Precision: the decisions are taken in fp32 as the GPU takes them: gq*inv_bs, *s
 * and +u are separate fp32 operations (no fused multiply-add); the mean is an fp64
 * sum of the fp32 products, divided by n in fp64 and rounded to fp32; s is an fp32
 * division.
 *
 * Counter RNG (splitmix64, Steele, Lea and Flood, OOPSLA 2014): mix is the
 * splitmix64 output function, G = 0x9E3779B97F4A7C15, key = mix(seed ^ (counter*G)),
 * u(j) = (mix(key + (j+1)*G) >> 40) * 2^-24 for global element index j = idx_base + i.
 */
uint64_t or_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

#define OR_G 0x9E3779B97F4A7C15ULL

float or_sr4_uniform(uint64_t seed, uint64_t counter, uint64_t j) {
    uint64_t key = or_mix64(seed ^ (counter * OR_G));
    uint64_t d = or_mix64(key + (j + 1) * OR_G);
    return (float)(d >> 40) * (1.0f / 16777216.0f);
}

float or_sr4_scale(const float* gq, int64_t n, float inv_bs, float target_step) {
    double sum = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        float g = gq[i] * inv_bs;
        sum += fabs((double)g);
    }
    float mean = n > 0 ? (float)(sum / (double)n) : 0.0f;
    if (!(mean > 0.0f) || !isfinite(mean)) return 0.0f;
    return target_step / mean;
}

void or_sr4_update(const int8_t* q, const float* gq, int64_t n, float inv_bs, float s, uint64_t seed,
                   int64_t idx_base, uint64_t counter, int clamp, int dither, int8_t* q_out, float* y_out) {
    for (int64_t i = 0; i < n; ++i) {
        float x = (gq[i] * inv_bs) * s;
        float u = dither ? or_sr4_uniform(seed, counter, (uint64_t)(idx_base + i)) : 0.5f;
        float y = x + u;
        if (y_out) y_out[i] = y;
        int v = q[i];
        if (isfinite(y)) {
            float d = floorf(y);
            if (d > 300.0f) d = 300.0f;
            if (d < -300.0f) d = -300.0f;
            v = or_clamp(v - (int)d, clamp);
        }
        q_out[i] = (int8_t)v;
    }
}

/* ------------------------------------------------------------ gradient norm, clip, skip */

/*
 * Global gradient L2 over several tensors and the clip / skip rule around AdamW
 * (page "train_gpu.cu": grad_l2_gpu sums squares over every parameter gradient in
 * double; page "nvg_train.rs": grad_norm is NaN/inf when a gradient is, and adam
 * multiplies the gradients by gmul; page "heal_gpu.rs": a non-finite norm skips the
 * step, otherwise gmul = clip / gn when gn > clip, else 1).
 *   or_sumsq       sum_i g_i^2 in fp64, ascending i
 *   or_clip_factor -1 when sqrt(sumsq) is not finite (skip the step); otherwise
 *                  max_norm / norm when max_norm > 0 and norm > max_norm, else 1
 */
double or_sumsq(const float* g, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += (double)g[i] * (double)g[i];
    return s;
}

double or_clip_factor(double sumsq, double max_norm) {
    double norm = sqrt(sumsq);
    if (!isfinite(norm)) return -1.0;
    if (max_norm > 0.0 && norm > max_norm) return max_norm / norm;
    return 1.0;
}

/* ------------------------------------------------------------ SR4 health panel */

/*
 * The SR4 health panel of one weight (page "train_gpu.cu", sr4_panel_compute,
 * computed from the post-step q and scale):
 *   counts[0..5] = #ternary -1, #ternary 0, #ternary +1, #|q| == clamp (rail),
 *                  #|q| < theta (dead), #ternary differing from the previous
 *                  ternary (churn; 0 when q_prev is NULL)
 *   sstats[0..2] = min, mean, max of scale over the N columns (mean in fp64).
 */
void or_sr4_panel(const int8_t* q, const int8_t* q_prev, const float* scale, int64_t K, int64_t N, int theta,
                  int clamp, uint64_t* counts, double* sstats) {
    for (int k = 0; k < 6; ++k) counts[k] = 0;
    for (int64_t i = 0; i < K * N; ++i) {
        int w = or_ternary(q[i], theta);
        int a = q[i] < 0 ? -q[i] : q[i];
        counts[w + 1] += 1;
        if (a == clamp) counts[3] += 1;
        if (a < theta) counts[4] += 1;
        if (q_prev && or_ternary(q_prev[i], theta) != w) counts[5] += 1;
    }
    double mn = 0.0, mx = 0.0, sum = 0.0;
    for (int64_t c = 0; c < N; ++c) {
        double s = (double)scale[c];
        if (c == 0 || s < mn) mn = s;
        if (c == 0 || s > mx) mx = s;
        sum += s;
    }
    sstats[0] = mn;
    sstats[1] = N > 0 ? sum / (double)N : 0.0;
    sstats[2] = mx;
}
