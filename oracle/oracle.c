/*
 * oracle.c -- plain, slow, CPU reference for the KOSMOS fused operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA path (comm_persistent_gemm_gb300/csrc).
 *
 * Every floating-point result is accumulated in IEEE double from the same bf16
 * (or MXFP8-quantised) inputs the GPU receives; outputs are NOT rounded to
 * bf16.  Loops follow the definitions with no blocking, fusion or reordering
 * of a sum: each output element is summed over K in ascending order (and, for
 * the reduce-scatter, over ranks r = 0..P-1 in that order).
 *
 * Sources (web pages on "KOSMOS: Self-scheduling Persistent Kernels for
 * Communication-Compute Overlap"):
 *   [explainer]  learnaivisually.com "KOSMOS -- Self-scheduling persistent
 *                kernels -- What does it mean?", paragraphs named by their
 *                opening words ("Start with the problem", "KOSMOS removes the
 *                manager", "Role switching only works", ...).
 *   [abstract]   the authors' arXiv abstract (2611.07477v1).
 *
 * Parity pins live in tests/test_oracle_*.py.  Functions whose exact values
 * have no independent pin are marked "parity unpinned" below (none at
 * present: every function has at least one pin).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32 word. */
ORC_EXPORT double orc_bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinity;
 * largest finite 1.75 * 2^8 = 448. */
ORC_EXPORT double orc_e4m3_to_f64(uint8_t q) {
    int s = (q >> 7) & 1;
    int e = (q >> 3) & 15;
    int m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 value, ties to even mantissa, saturating to +-448 (the
 * quantiser below never reaches the saturation branch: its scale keeps every
 * scaled element within +-448). */
ORC_EXPORT uint8_t orc_f64_to_e4m3(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid: multiples of 2^-9; 8 * 2^-9 is the smallest normal,
         * whose code (exponent 1, mantissa 0) is also the integer 8 */
        double mq = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)mq);
    }
    int ex;
    frexp(a, &ex);               /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;              /* a = (1 + t) * 2^E, t in [0, 1) */
    double t = a / ldexp(1.0, E) - 1.0;
    double mq = nearbyint(t * 8.0);
    if (mq == 8.0) { mq = 0.0; E += 1; }
    int be = E + 7;
    if (be > 15 || (be == 15 && mq == 7.0)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)(be << 3) | (uint8_t)mq);
}

/* Shared exponent of one 32-element block: the smallest integer e with
 * blockmax <= 448 * 2^e (that is, 2^ceil(log2(blockmax / 448))), clamped to the
 * E8M0 range [-127, 127].  An all-zero block takes e = 0. */
ORC_EXPORT int orc_mx_scale_exp(double blockmax) {
    if (!(blockmax > 0.0)) return 0;
    int e = (int)ceil(log2(blockmax / 448.0));
    while (blockmax > ldexp(448.0, e)) e++;
    while (blockmax <= ldexp(448.0, e - 1)) e--;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* MXFP8 quantisation of a row-major bf16 matrix [rows, cols].
 *   along_cols = 1: blocks are 32 contiguous columns of one row (an activation
 *                   X[m, K]); scales are [rows, cols/32].
 *   along_cols = 0: blocks are 32 contiguous rows of one column (a weight
 *                   W[K, n]); scales are [cols, rows/32].
 * q keeps the input's [rows, cols] layout.  Scale byte = e + 127 (E8M0). */
ORC_EXPORT int orc_mxfp8_quantize(int64_t rows, int64_t cols, const uint16_t *x,
                                  int along_cols, uint8_t *q, uint8_t *scales) {
    if (along_cols) {
        if (cols % 32) return 1;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < rows; i++)
            for (int64_t b = 0; b < cols / 32; b++) {
                double mx = 0.0;
                for (int j = 0; j < 32; j++) {
                    double a = fabs(orc_bf16_to_f64(x[i * cols + b * 32 + j]));
                    if (a > mx) mx = a;
                }
                int e = orc_mx_scale_exp(mx);
                scales[i * (cols / 32) + b] = (uint8_t)(e + 127);
                for (int j = 0; j < 32; j++) {
                    double v = orc_bf16_to_f64(x[i * cols + b * 32 + j]);
                    q[i * cols + b * 32 + j] = orc_f64_to_e4m3(ldexp(v, -e));
                }
            }
    } else {
        if (rows % 32) return 1;
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; c++)
            for (int64_t b = 0; b < rows / 32; b++) {
                double mx = 0.0;
                for (int j = 0; j < 32; j++) {
                    double a = fabs(orc_bf16_to_f64(x[(b * 32 + j) * cols + c]));
                    if (a > mx) mx = a;
                }
                int e = orc_mx_scale_exp(mx);
                scales[c * (rows / 32) + b] = (uint8_t)(e + 127);
                for (int j = 0; j < 32; j++) {
                    double v = orc_bf16_to_f64(x[(b * 32 + j) * cols + c]);
                    q[(b * 32 + j) * cols + c] = orc_f64_to_e4m3(ldexp(v, -e));
                }
            }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* All-gather + GEMM                                                         */
/* ------------------------------------------------------------------------ */

/* [explainer, "Start with the problem"]: each layer gathers the pieces of its
 * input from the other ranks before the matrix multiplication.  The gathered
 * input is the row concatenation [X_0; X_1; ...; X_{P-1}] and
 *     Y = concat_r(X_r) . W,      X_r: [m, k],  W: [k, n],  Y: [P*m, n].
 * rows: global row indices of Y to compute (NULL -> all P*m rows, in order);
 * y: [nrows, n] doubles. */
ORC_EXPORT int orc_ag_gemm(int P, int64_t m, int64_t k, int64_t n,
                           const uint16_t *const *x, const uint16_t *w,
                           const int64_t *rows, int64_t nrows, double *y) {
    if (!rows) nrows = (int64_t)P * m;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(k * n));
    if (!wd) return 2;
    for (int64_t i = 0; i < k * n; i++) wd[i] = orc_bf16_to_f64(w[i]);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nrows; t++) {
        int64_t g = rows ? rows[t] : t;
        if (g < 0 || g >= (int64_t)P * m) { bad = 1; continue; }
        int64_t r = g / m, i = g % m;
        const uint16_t *xr = x[r] + i * k;
        double *acc = y + t * n;
        for (int64_t j = 0; j < n; j++) acc[j] = 0.0;
        for (int64_t kk = 0; kk < k; kk++) {
            double a = orc_bf16_to_f64(xr[kk]);
            const double *wrow = wd + kk * n;
            for (int64_t j = 0; j < n; j++) acc[j] += a * wrow[j];
        }
    }
    free(wd);
    return bad ? 1 : 0;
}

/* The MXFP8 variant [abstract: "1.10-1.25x in MXFP8"]: the same product on the
 * dequantised operands, X_q[i][kk] = e4m3(qx) * 2^(sx[i][kk/32] - 127) and
 * W_q[kk][j] = e4m3(qw) * 2^(sw[j][kk/32] - 127), both exact in double.
 * Scale layouts: sx_r [m, k/32], sw [n, k/32]. */
ORC_EXPORT int orc_ag_gemm_mxfp8(int P, int64_t m, int64_t k, int64_t n,
                                 const uint8_t *const *qx, const uint8_t *const *sx,
                                 const uint8_t *qw, const uint8_t *sw,
                                 const int64_t *rows, int64_t nrows, double *y) {
    if (k % 32) return 1;
    if (!rows) nrows = (int64_t)P * m;
    int64_t kb = k / 32;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(k * n));
    if (!wd) return 2;
    for (int64_t kk = 0; kk < k; kk++)
        for (int64_t j = 0; j < n; j++)
            wd[kk * n + j] = ldexp(orc_e4m3_to_f64(qw[kk * n + j]), (int)sw[j * kb + kk / 32] - 127);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nrows; t++) {
        int64_t g = rows ? rows[t] : t;
        if (g < 0 || g >= (int64_t)P * m) { bad = 1; continue; }
        int64_t r = g / m, i = g % m;
        double *acc = y + t * n;
        for (int64_t j = 0; j < n; j++) acc[j] = 0.0;
        for (int64_t kk = 0; kk < k; kk++) {
            double a = ldexp(orc_e4m3_to_f64(qx[r][i * k + kk]), (int)sx[r][i * kb + kk / 32] - 127);
            const double *wrow = wd + kk * n;
            for (int64_t j = 0; j < n; j++) acc[j] += a * wrow[j];
        }
    }
    free(wd);
    return bad ? 1 : 0;
}

/* ------------------------------------------------------------------------ */
/* GEMM + reduce-scatter                                                     */
/* ------------------------------------------------------------------------ */

/* [explainer, "Start with the problem"]: after the multiplication each rank
 * holds a partial result; the partials are scattered and added.  With rank r
 * holding X_r [m, k] and W_r [k, n]:
 *     Y = sum_{r=0..P-1} X_r . W_r   (summed in rank order),
 * and rank c receives chunk c = rows [c*m/P, (c+1)*m/P) of Y.
 * rows: global rows of Y (NULL -> all m); y: [nrows, n]. */
ORC_EXPORT int orc_gemm_rs(int P, int64_t m, int64_t k, int64_t n,
                           const uint16_t *const *x, const uint16_t *const *w,
                           const int64_t *rows, int64_t nrows, double *y) {
    if (!rows) nrows = m;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(P * k * n));
    if (!wd) return 2;
    for (int r = 0; r < P; r++)
        for (int64_t i = 0; i < k * n; i++) wd[(int64_t)r * k * n + i] = orc_bf16_to_f64(w[r][i]);
    int bad = 0;
#pragma omp parallel
    {
        double *part = (double *)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < nrows; t++) {
            int64_t g = rows ? rows[t] : t;
            if (g < 0 || g >= m || !part) { bad = 1; continue; }
            double *acc = y + t * n;
            for (int64_t j = 0; j < n; j++) acc[j] = 0.0;
            for (int r = 0; r < P; r++) {
                const uint16_t *xr = x[r] + g * k;
                for (int64_t j = 0; j < n; j++) part[j] = 0.0;
                for (int64_t kk = 0; kk < k; kk++) {
                    double a = orc_bf16_to_f64(xr[kk]);
                    const double *wrow = wd + (int64_t)r * k * n + kk * n;
                    for (int64_t j = 0; j < n; j++) part[j] += a * wrow[j];
                }
                for (int64_t j = 0; j < n; j++) acc[j] += part[j];
            }
        }
        free(part);
    }
    free(wd);
    return bad ? 1 : 0;
}

/* MXFP8 GEMM + reduce-scatter [abstract: the MXFP8 results cover the whole
 * TP+SP layer; same definition as orc_gemm_rs]: Y = sum_r dequant(X_r) .
 * dequant(W_r), each element e4m3 x 2^(scale - 127) exactly in fp64; X_r
 * scales [m, k/32] (one per row and 32 K), W_r scales [n, k/32] (one per
 * column and 32 K), row-major.  Ranks summed in order 0..P-1 per row. */
ORC_EXPORT int orc_gemm_rs_mxfp8(int P, int64_t m, int64_t k, int64_t n,
                                 const uint8_t *const *qx, const uint8_t *const *sx,
                                 const uint8_t *const *qw, const uint8_t *const *sw,
                                 const int64_t *rows, int64_t nrows, double *y) {
    if (k % 32) return 1;
    if (!rows) nrows = m;
    int64_t kb = k / 32;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(P * k * n));
    if (!wd) return 2;
    for (int r = 0; r < P; r++)
        for (int64_t kk = 0; kk < k; kk++)
            for (int64_t j = 0; j < n; j++)
                wd[(int64_t)r * k * n + kk * n + j] =
                    ldexp(orc_e4m3_to_f64(qw[r][kk * n + j]), (int)sw[r][j * kb + kk / 32] - 127);
    int bad = 0;
#pragma omp parallel
    {
        double *part = (double *)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < nrows; t++) {
            int64_t g = rows ? rows[t] : t;
            if (g < 0 || g >= m || !part) { bad = 1; continue; }
            double *acc = y + t * n;
            for (int64_t j = 0; j < n; j++) acc[j] = 0.0;
            for (int r = 0; r < P; r++) {
                for (int64_t j = 0; j < n; j++) part[j] = 0.0;
                for (int64_t kk = 0; kk < k; kk++) {
                    double a = ldexp(orc_e4m3_to_f64(qx[r][g * k + kk]), (int)sx[r][g * kb + kk / 32] - 127);
                    const double *wrow = wd + (int64_t)r * k * n + kk * n;
                    for (int64_t j = 0; j < n; j++) part[j] += a * wrow[j];
                }
                for (int64_t j = 0; j < n; j++) acc[j] += part[j];
            }
        }
        free(part);
    }
    free(wd);
    return bad ? 1 : 0;
}

/* ------------------------------------------------------------------------ */
/* MoE expert layer (forward)                                                */
/* ------------------------------------------------------------------------ */

/* Top-k of one row of scores: the k largest values, emitted in descending
 * order; equal values are ordered by the lower index first.  Selection on the
 * logits equals selection on the softmax probabilities (softmax is strictly
 * increasing in each logit). */
static void orc_topk_row(int E, int K, const double *s, int32_t *idx) {
    char *taken = (char *)calloc((size_t)E, 1);
    for (int kk = 0; kk < K; kk++) {
        int best = -1;
        for (int e = 0; e < E; e++) {
            if (taken[e]) continue;
            if (best < 0 || s[e] > s[best]) best = e;   /* strict: ties keep the lower index */
        }
        idx[kk] = best;
        taken[best] = 1;
    }
    free(taken);
}

/* Top-k over float32 scores (used to check the kernel's index decisions in
 * the kernel's own precision: the comparison of two floats is exact in
 * double). */
ORC_EXPORT int orc_topk_f32(int64_t T, int E, int K, const float *scores, int32_t *idx) {
    if (K < 1 || K > E) return 1;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp for
        for (int64_t t = 0; t < T; t++) {
            for (int e = 0; e < E; e++) s[e] = (double)scores[t * E + e];
            orc_topk_row(E, K, s, idx + t * K);
        }
        free(s);
    }
    return 0;
}

/* Expert-parallel dispatch tables [explainer, "Start with the problem": the
 * all-to-all sends each token to the rank holding its expert].  Given the
 * top-k indices:
 *   counts[e]   = number of (t, k) slots routed to expert e;
 *   offsets[e]  = exclusive prefix sum of counts in expert order (expert e of
 *                 rank q = e / (E/P) is received contiguously, experts in
 *                 ascending order, so rank q's receive buffer is a contiguous
 *                 slice);
 *   pos[t][k]   = offsets[e] + #{t' < t routed to e}  (receive order: expert
 *                 ascending, then token ascending). */
ORC_EXPORT int orc_moe_dispatch_tables(int64_t T, int E, int K, const int32_t *idx,
                                       int32_t *counts, int32_t *offsets, int32_t *pos) {
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (int64_t i = 0; i < T * K; i++) {
        if (idx[i] < 0 || idx[i] >= E) return 1;
        counts[idx[i]]++;
    }
    int32_t run = 0;
    for (int e = 0; e < E; e++) { offsets[e] = run; run += counts[e]; }
    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; t++)
        for (int kk = 0; kk < K; kk++) {
            int e = idx[t * K + kk];
            pos[t * K + kk] = offsets[e] + seen[e]++;
        }
    free(seen);
    return 0;
}

/* Router [abstract: "an entire expert layer, from router to fold"]:
 *   logits = X . W_router                  (fp64)
 *   p      = softmax(logits) over experts  (fp64)
 *   idx    = top-K of the logits (ties to the lower expert index), emitted in
 *            descending order
 *   gate_k = p[idx_k] / sum_{j<K} p[idx_j]  (renormalised over the top-K)
 * followed by the dispatch tables above. */
ORC_EXPORT int orc_moe_route(int64_t T, int64_t H, int E, int K,
                             const uint16_t *x, const uint16_t *wr,
                             double *logits, int32_t *idx, double *gate,
                             int32_t *counts, int32_t *offsets, int32_t *pos) {
    if (K < 1 || K > E) return 1;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(H * E));
    if (!wd) return 2;
    for (int64_t i = 0; i < H * E; i++) wd[i] = orc_bf16_to_f64(wr[i]);
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < T; t++) {
            double *l = logits + t * E;
            for (int e = 0; e < E; e++) l[e] = 0.0;
            for (int64_t h = 0; h < H; h++) {
                double a = orc_bf16_to_f64(x[t * H + h]);
                for (int e = 0; e < E; e++) l[e] += a * wd[h * E + e];
            }
            double mx = l[0];
            for (int e = 1; e < E; e++) if (l[e] > mx) mx = l[e];
            double z = 0.0;
            for (int e = 0; e < E; e++) { p[e] = exp(l[e] - mx); z += p[e]; }
            for (int e = 0; e < E; e++) p[e] /= z;
            orc_topk_row(E, K, l, idx + t * K);
            double zs = 0.0;
            for (int kk = 0; kk < K; kk++) zs += p[idx[t * K + kk]];
            for (int kk = 0; kk < K; kk++) gate[t * K + kk] = p[idx[t * K + kk]] / zs;
        }
        free(p);
    }
    free(wd);
    return orc_moe_dispatch_tables(T, E, K, idx, counts, offsets, pos);
}

/* SwiGLU expert, gate input first: silu(a) = a / (1 + exp(-a)). */
static double orc_silu(double a) { return a / (1.0 + exp(-a)); }

/* Expert computation and gate-weighted combine ("fold") for selected tokens:
 *   out[t] = sum_{k<K} gate[t][k] * ( silu(x_t W_g[e]) * (x_t W_u[e]) ) W_d[e],
 *            e = idx[t][k], summed in k order.
 * Weights per EP rank q (experts q*Eq .. q*Eq+Eq-1):
 *   wg[q], wu[q]: [Eq, H, I];  wd[q]: [Eq, I, H].
 * identity != 0 replaces every expert by the identity map (out[t] = x_t *
 * sum_k gate[t][k]), the check named by the method's description.
 * tokens: token indices (NULL -> all T); out: [ntok, H]. */
ORC_EXPORT int orc_moe_experts(int64_t T, int64_t H, int E, int K, int64_t I, int P,
                               const uint16_t *x, const int32_t *idx, const double *gate,
                               const uint16_t *const *wg, const uint16_t *const *wu,
                               const uint16_t *const *wd, int identity,
                               const int64_t *tokens, int64_t ntok, double *out) {
    if (E % P) return 1;
    int Eq = E / P;
    if (!tokens) ntok = T;
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < ntok; s++) {
            int64_t t = tokens ? tokens[s] : s;
            if (t < 0 || t >= T) { bad = 1; continue; }
            double *o = out + s * H;
            for (int64_t h = 0; h < H; h++) { xt[h] = orc_bf16_to_f64(x[t * H + h]); o[h] = 0.0; }
            for (int kk = 0; kk < K; kk++) {
                int e = idx[t * K + kk];
                double gk = gate[t * K + kk];
                if (identity) {
                    for (int64_t h = 0; h < H; h++) o[h] += gk * xt[h];
                    continue;
                }
                int q = e / Eq, le = e % Eq;
                const uint16_t *Wg = wg[q] + (int64_t)le * H * I;
                const uint16_t *Wu = wu[q] + (int64_t)le * H * I;
                const uint16_t *Wd = wd[q] + (int64_t)le * I * H;
                for (int64_t i = 0; i < I; i++) { g[i] = 0.0; u[i] = 0.0; }
                for (int64_t h = 0; h < H; h++) {
                    double a = xt[h];
                    for (int64_t i = 0; i < I; i++) {
                        g[i] += a * orc_bf16_to_f64(Wg[h * I + i]);
                        u[i] += a * orc_bf16_to_f64(Wu[h * I + i]);
                    }
                }
                for (int64_t hh = 0; hh < H; hh++) y[hh] = 0.0;
                for (int64_t i = 0; i < I; i++) {
                    double hv = orc_silu(g[i]) * u[i];
                    for (int64_t hh = 0; hh < H; hh++) y[hh] += hv * orc_bf16_to_f64(Wd[i * H + hh]);
                }
                for (int64_t hh = 0; hh < H; hh++) o[hh] += gk * y[hh];
            }
        }
        free(xt); free(g); free(u); free(y);
    }
    return bad ? 1 : 0;
}

/* MXFP8 experts [abstract: the MXFP8 results; reading: an MXFP8 expert layer
 * quantises what enters each expert GEMM].  The same layer as orc_moe_experts
 * with every GEMM operand in MXFP8:
 *   x_t      : e4m3 codes xq[t][h] x 2^(xs[t][h/32] - 127)   (the token rows,
 *              quantised once along the hidden dimension);
 *   W_g[e], W_u[e] [H, I]: codes x 2^(scale[i][h/32] - 127);
 *   W_d[e] [I, H]       : codes x 2^(scale[h][i/32] - 127);
 *   g, u = x_t W_g, x_t W_u (fp64 sums of exact products); h = silu(g) * u;
 *   h quantised along I in blocks of 32 by the same rule as the inputs
 *   (e = smallest integer with blockmax <= 448 * 2^e, codes = E4M3 RNE of
 *   h / 2^e), then y = dequant(h) W_d and out[t] = sum_k gate * y in k order.
 * Weight scales per EP rank q: Eq experts' row-major blocks one after the
 * other ([Eq][I][H/32] for gate and up, [Eq][H][I/32] for down). */
ORC_EXPORT int orc_moe_experts_mxfp8(int64_t T, int64_t H, int E, int K, int64_t I, int P,
                                     const uint8_t *xq, const uint8_t *xs, const int32_t *idx,
                                     const double *gate,
                                     const uint8_t *const *wgq, const uint8_t *const *wgs,
                                     const uint8_t *const *wuq, const uint8_t *const *wus,
                                     const uint8_t *const *wdq, const uint8_t *const *wds,
                                     const int64_t *tokens, int64_t ntok, double *out) {
    if (E % P || H % 32 || I % 32) return 1;
    int Eq = E / P;
    if (!tokens) ntok = T;
    double code[256], pw[256];
    for (int c = 0; c < 256; c++) { code[c] = orc_e4m3_to_f64((uint8_t)c); pw[c] = ldexp(1.0, c - 127); }
    const int64_t HB = H / 32, IB = I / 32;
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *hd = (double *)malloc(sizeof(double) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < ntok; s++) {
            int64_t t = tokens ? tokens[s] : s;
            if (t < 0 || t >= T) { bad = 1; continue; }
            double *o = out + s * H;
            for (int64_t h = 0; h < H; h++) {
                xt[h] = code[xq[t * H + h]] * pw[xs[t * HB + h / 32]];
                o[h] = 0.0;
            }
            for (int kk = 0; kk < K; kk++) {
                int e = idx[t * K + kk];
                int q = e / Eq, le = e % Eq;
                const uint8_t *Qg = wgq[q] + (int64_t)le * H * I, *Sg = wgs[q] + (int64_t)le * I * HB;
                const uint8_t *Qu = wuq[q] + (int64_t)le * H * I, *Su = wus[q] + (int64_t)le * I * HB;
                const uint8_t *Qd = wdq[q] + (int64_t)le * I * H, *Sd = wds[q] + (int64_t)le * H * IB;
                for (int64_t i = 0; i < I; i++) { g[i] = 0.0; u[i] = 0.0; }
                for (int64_t h = 0; h < H; h++) {
                    double a = xt[h];
                    for (int64_t i = 0; i < I; i++) {
                        g[i] += a * (code[Qg[h * I + i]] * pw[Sg[i * HB + h / 32]]);
                        u[i] += a * (code[Qu[h * I + i]] * pw[Su[i * HB + h / 32]]);
                    }
                }
                for (int64_t b = 0; b < IB; b++) {
                    double hv[32], mx = 0.0;
                    for (int j = 0; j < 32; j++) {
                        hv[j] = orc_silu(g[b * 32 + j]) * u[b * 32 + j];
                        if (fabs(hv[j]) > mx) mx = fabs(hv[j]);
                    }
                    int ex = orc_mx_scale_exp(mx);
                    for (int j = 0; j < 32; j++)
                        hd[b * 32 + j] = ldexp(orc_e4m3_to_f64(orc_f64_to_e4m3(ldexp(hv[j], -ex))), ex);
                }
                for (int64_t hh = 0; hh < H; hh++) y[hh] = 0.0;
                for (int64_t i = 0; i < I; i++) {
                    double hv = hd[i];
                    for (int64_t hh = 0; hh < H; hh++) y[hh] += hv * (code[Qd[i * H + hh]] * pw[Sd[hh * IB + i / 32]]);
                }
                double gk = gate[t * K + kk];
                for (int64_t hh = 0; hh < H; hh++) o[hh] += gk * y[hh];
            }
        }
        free(xt); free(g); free(u); free(hd); free(y);
    }
    return bad ? 1 : 0;
}

/* ------------------------------------------------------------------------ */
/* MoE expert layer (backward)                                               */
/* ------------------------------------------------------------------------ */
/* [abstract: "one launch per direction"; reading: the gradients of the
 * forward layer above with the routing (top-K indices) held fixed].  Forward:
 *   l_t = x_t Wr, p_t = softmax(l_t), S_t = sum_{k<K} p_t[e_k],
 *   gate_{t,k} = p_t[e_k] / S_t, g = x_t Wg[e], u = x_t Wu[e],
 *   h = silu(g) * u, y_{t,k} = h Wd[e], out_t = sum_k gate_{t,k} y_{t,k}.
 * Given dout_t = dL/dout_t:
 *   dgate_{t,k} = <dout_t, y_{t,k}>,  dy_{t,k} = gate_{t,k} dout_t,
 *   dh = dy Wd[e]^T,  dg = dh * u * silu'(g),  du = dh * silu(g),
 *   silu'(g) = s (1 + g (1 - s)), s = 1 / (1 + exp(-g)),
 *   dp_j = (dgate_{k(j)} - sum_k dgate_k gate_k) / S for j = e_{k(j)} in the
 *   top-K set, 0 elsewhere;  dl = p * (dp - <p, dp>),
 *   dx_t = sum_k (dg Wg[e]^T + du Wu[e]^T) + dl_t Wr^T,
 *   dWg[e] = sum over slots routed to e of x_t^T dg, dWu[e] likewise with du,
 *   dWd[e] = sum of h^T dy,  dWr = sum_t x_t^T dl_t.
 * All in fp64 from the bf16 inputs; logits from orc_moe_route (fp64). */

typedef struct {
    int64_t H, I;
    const uint16_t *Wg, *Wu, *Wd;
} orc_expert_w;

/* One slot: forward g, u, h, y and backward dg, du for a token row xt
 * (fp64) and upstream dy_row = gate * dout (fp64). */
static void orc_slot_fwd_bwd(const orc_expert_w *w, const double *xt, const double *dyv, double *g, double *u,
                             double *hh, double *y, double *dh, double *dg, double *du) {
    int64_t H = w->H, I = w->I;
    for (int64_t i = 0; i < I; i++) { g[i] = 0.0; u[i] = 0.0; }
    for (int64_t h = 0; h < H; h++) {
        double a = xt[h];
        for (int64_t i = 0; i < I; i++) {
            g[i] += a * orc_bf16_to_f64(w->Wg[h * I + i]);
            u[i] += a * orc_bf16_to_f64(w->Wu[h * I + i]);
        }
    }
    for (int64_t i = 0; i < I; i++) hh[i] = orc_silu(g[i]) * u[i];
    if (y) {
        for (int64_t c = 0; c < H; c++) y[c] = 0.0;
        for (int64_t i = 0; i < I; i++)
            for (int64_t c = 0; c < H; c++) y[c] += hh[i] * orc_bf16_to_f64(w->Wd[i * H + c]);
    }
    for (int64_t i = 0; i < I; i++) {
        double acc = 0.0;
        for (int64_t c = 0; c < H; c++) acc += dyv[c] * orc_bf16_to_f64(w->Wd[i * H + c]);
        dh[i] = acc;
        double sg = 1.0 / (1.0 + exp(-g[i]));
        dg[i] = dh[i] * u[i] * sg * (1.0 + g[i] * (1.0 - sg));
        du[i] = dh[i] * orc_silu(g[i]);
    }
}

static orc_expert_w orc_expert(int e, int Eq, int64_t H, int64_t I, const uint16_t *const *wg,
                               const uint16_t *const *wu, const uint16_t *const *wd) {
    orc_expert_w w;
    int q = e / Eq, le = e % Eq;
    w.H = H; w.I = I;
    w.Wg = wg[q] + (int64_t)le * H * I;
    w.Wu = wu[q] + (int64_t)le * H * I;
    w.Wd = wd[q] + (int64_t)le * I * H;
    return w;
}

/* Router backward of one token from its dgate: dl[E] (see above). */
static void orc_router_bwd(int E, int K, const double *l, const int32_t *idx, const double *dgate, double *dl) {
    double mx = l[0];
    for (int e = 1; e < E; e++) if (l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; e++) { dl[e] = exp(l[e] - mx); z += dl[e]; }
    for (int e = 0; e < E; e++) dl[e] /= z;  /* p */
    double S = 0.0;
    for (int k = 0; k < K; k++) S += dl[idx[k]];
    double sdg = 0.0;
    for (int k = 0; k < K; k++) sdg += dgate[k] * dl[idx[k]] / S;
    /* dp is nonzero on the top-K set only */
    double pdp = 0.0;
    for (int k = 0; k < K; k++) pdp += dl[idx[k]] * (dgate[k] - sdg) / S;
    double *p = dl;  /* overwritten in place below: keep dp of the top-K in a small table */
    double dpk[64];
    for (int k = 0; k < K; k++) dpk[k] = (dgate[k] - sdg) / S;
    for (int e = 0; e < E; e++) {
        double dp = 0.0;
        for (int k = 0; k < K; k++) if (idx[k] == e) dp = dpk[k];
        p[e] = p[e] * (dp - pdp);
    }
}

/* dx of selected tokens (the expert and router paths), with dgate [ntok, K]
 * and dl [ntok, E] of those tokens.  logits: [T, E] fp64 from orc_moe_route. */
ORC_EXPORT int orc_moe_bwd_tokens(int64_t T, int64_t H, int E, int K, int64_t I, int P,
                                  const uint16_t *x, const uint16_t *wr, const double *logits,
                                  const int32_t *idx, const double *gate, const uint16_t *dout,
                                  const uint16_t *const *wg, const uint16_t *const *wu,
                                  const uint16_t *const *wd, const int64_t *tokens, int64_t ntok,
                                  double *dx, double *dgate_out, double *dl_out) {
    if (E % P || K > 64) return 1;
    int Eq = E / P;
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *dv = (double *)malloc(sizeof(double) * (size_t)H);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *hh = (double *)malloc(sizeof(double) * (size_t)I);
        double *dh = (double *)malloc(sizeof(double) * (size_t)I);
        double *dg = (double *)malloc(sizeof(double) * (size_t)I);
        double *du = (double *)malloc(sizeof(double) * (size_t)I);
        double *dl = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < ntok; s++) {
            int64_t t = tokens ? tokens[s] : s;
            if (t < 0 || t >= T) { bad = 1; continue; }
            double *o = dx + s * H;
            double dgt[64];
            for (int64_t c = 0; c < H; c++) { xt[c] = orc_bf16_to_f64(x[t * H + c]); o[c] = 0.0; }
            for (int k = 0; k < K; k++) {
                int e = idx[t * K + k];
                orc_expert_w w = orc_expert(e, Eq, H, I, wg, wu, wd);
                double gk = gate[t * K + k];
                for (int64_t c = 0; c < H; c++) dv[c] = gk * orc_bf16_to_f64(dout[t * H + c]);
                orc_slot_fwd_bwd(&w, xt, dv, g, u, hh, y, dh, dg, du);
                double acc = 0.0;
                for (int64_t c = 0; c < H; c++) acc += orc_bf16_to_f64(dout[t * H + c]) * y[c];
                dgt[k] = acc;
                for (int64_t c = 0; c < H; c++) {
                    double a = 0.0;
                    for (int64_t i = 0; i < I; i++)
                        a += dg[i] * orc_bf16_to_f64(w.Wg[c * I + i]) + du[i] * orc_bf16_to_f64(w.Wu[c * I + i]);
                    o[c] += a;
                }
            }
            orc_router_bwd(E, K, logits + t * E, idx + t * K, dgt, dl);
            for (int64_t c = 0; c < H; c++) {
                double a = 0.0;
                for (int e = 0; e < E; e++) a += dl[e] * orc_bf16_to_f64(wr[c * E + e]);
                o[c] += a;
            }
            if (dgate_out) for (int k = 0; k < K; k++) dgate_out[s * K + k] = dgt[k];
            if (dl_out) for (int e = 0; e < E; e++) dl_out[s * E + e] = dl[e];
        }
        free(xt); free(dv); free(y); free(g); free(u); free(hh); free(dh); free(dg); free(du); free(dl);
    }
    return bad ? 1 : 0;
}

/* Weight gradients of selected experts: dwg, dwu [nexp, H, I], dwd [nexp, I, H];
 * sums over the slots routed to each expert in (token, k) order. */
ORC_EXPORT int orc_moe_bwd_experts(int64_t T, int64_t H, int E, int K, int64_t I, int P,
                                   const uint16_t *x, const int32_t *idx, const double *gate,
                                   const uint16_t *dout, const uint16_t *const *wg,
                                   const uint16_t *const *wu, const uint16_t *const *wd,
                                   const int32_t *experts, int nexp, double *dwg, double *dwu, double *dwd) {
    if (E % P) return 1;
    int Eq = E / P;
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *dv = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *hh = (double *)malloc(sizeof(double) * (size_t)I);
        double *dh = (double *)malloc(sizeof(double) * (size_t)I);
        double *dg = (double *)malloc(sizeof(double) * (size_t)I);
        double *du = (double *)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < nexp; n++) {
            int e = experts[n];
            if (e < 0 || e >= E) { bad = 1; continue; }
            orc_expert_w w = orc_expert(e, Eq, H, I, wg, wu, wd);
            double *Dg = dwg + (int64_t)n * H * I, *Du = dwu + (int64_t)n * H * I, *Dd = dwd + (int64_t)n * I * H;
            for (int64_t j = 0; j < H * I; j++) { Dg[j] = 0.0; Du[j] = 0.0; Dd[j] = 0.0; }
            for (int64_t t = 0; t < T; t++)
                for (int k = 0; k < K; k++) {
                    if (idx[t * K + k] != e) continue;
                    for (int64_t c = 0; c < H; c++) {
                        xt[c] = orc_bf16_to_f64(x[t * H + c]);
                        dv[c] = gate[t * K + k] * orc_bf16_to_f64(dout[t * H + c]);
                    }
                    orc_slot_fwd_bwd(&w, xt, dv, g, u, hh, NULL, dh, dg, du);
                    for (int64_t c = 0; c < H; c++)
                        for (int64_t i = 0; i < I; i++) {
                            Dg[c * I + i] += xt[c] * dg[i];
                            Du[c * I + i] += xt[c] * du[i];
                        }
                    for (int64_t i = 0; i < I; i++)
                        for (int64_t c = 0; c < H; c++) Dd[i * H + c] += hh[i] * dv[c];
                }
        }
        free(xt); free(dv); free(g); free(u); free(hh); free(dh); free(dg); free(du);
    }
    return bad ? 1 : 0;
}

/* dWr [H, E] = sum over all tokens of x_t^T dl_t (token order). */
ORC_EXPORT int orc_moe_bwd_router_weight(int64_t T, int64_t H, int E, int K, int64_t I, int P,
                                         const uint16_t *x, const uint16_t *wr, const double *logits,
                                         const int32_t *idx, const double *gate, const uint16_t *dout,
                                         const uint16_t *const *wg, const uint16_t *const *wu,
                                         const uint16_t *const *wd, double *dwr) {
    double *dx = (double *)malloc(sizeof(double) * (size_t)(T * H));
    double *dl = (double *)malloc(sizeof(double) * (size_t)(T * E));
    if (!dx || !dl) { free(dx); free(dl); return 2; }
    int rc = orc_moe_bwd_tokens(T, H, E, K, I, P, x, wr, logits, idx, gate, dout, wg, wu, wd, NULL, T, dx, NULL, dl);
    if (!rc) {
        for (int64_t j = 0; j < H * E; j++) dwr[j] = 0.0;
        for (int64_t t = 0; t < T; t++)
            for (int64_t c = 0; c < H; c++) {
                double a = orc_bf16_to_f64(x[t * H + c]);
                for (int e = 0; e < E; e++) dwr[c * E + e] += a * dl[t * E + e];
            }
    }
    free(dx); free(dl);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Work rails ("the order of the rail is the schedule")                      */
/* ------------------------------------------------------------------------ */
/* [explainer, "Role switching only works"]: data is produced in the order its
 * consumers claim it.  Entries are written as 4 int32 fields
 * {kind, a, b, c}; kinds: 1 TRANSFER(shard, piece, part), 2 TILE, 3 REDUCE,
 * 10 TILE_HALF (one half of a tile's K range).
 * Tile and piece heights are R rows; output tiles are BN columns wide. */

enum { ORC_TRANSFER = 1, ORC_TILE = 2, ORC_REDUCE = 3, ORC_TILE_HALF = 10 };

static int64_t orc_cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* All-gather rails.
 * Transfer rail: remote shards s = 1..P-1 in the order the multiplication
 * consumes them, each cut into pieces j of R rows; then the local shard's own
 * pieces (copied into the gathered buffer; nothing waits on them).  Each
 * piece is split into R / PR parts q of PR rows, in row order, so that
 * several movers can fill the piece the next tile waits for [the pages do
 * not fix the transfer granularity; a piece counts as arrived once all of
 * its parts have arrived].  Parts past the shard's last row are still
 * entries (empty ones).
 * Tile rail: output tiles TILE(shard, tile-row, tile-col) of TR rows and BN
 * columns, row-major over tile rows with the local shard (s = 0) first, then
 * s = 1, 2, ...  The last XS tiles of that order are each replaced by two
 * entries TILE_HALF(shard, tile-row, 2 * tile-col + h) that compute the
 * tile over the first (h = 0) and the second (h = 1) half of the K blocks;
 * the output of the tile is the sum of the two [the pages give no tile
 * shapes; halving the final wave's tiles shortens the tail, where CTAs that
 * drew one tile more than others would otherwise finish a whole tile
 * later.  Halving K keeps the operand bytes per multiply-add of a whole
 * tile, which halving the columns would not].
 * Returns the number of entries written (transfer rail then tile rail), or
 * the count only when out == NULL; -1 for inconsistent arguments. */
ORC_EXPORT int64_t orc_rail_ag(int P, int64_t m, int64_t n, int R, int BN, int TR, int PR, int64_t XS,
                               int32_t *transfer_out, int64_t *n_transfer,
                               int32_t *tile_out, int64_t *n_tile) {
    if (PR < 1 || R % PR != 0 || XS < 0 || BN % 2 != 0) return -1;
    int64_t pieces = orc_cdiv(m, R), tn = orc_cdiv(n, BN), tm = orc_cdiv(m, TR);
    int parts = R / PR;
    int64_t n_full = (int64_t)P * tm * tn;
    if (XS > n_full) XS = n_full;
    int64_t nt = 0, nb = 0;
    for (int s = 1; s <= P; s++) {
        int shard = (s == P) ? 0 : s;
        for (int64_t j = 0; j < pieces; j++)
            for (int q = 0; q < parts; q++) {
                if (transfer_out) {
                    int32_t *e = transfer_out + 4 * nt;
                    e[0] = ORC_TRANSFER; e[1] = shard; e[2] = (int32_t)j; e[3] = q;
                }
                nt++;
            }
    }
    int64_t f = 0; /* position of the tile in the unsplit order */
    for (int s = 0; s < P; s++)
        for (int64_t i = 0; i < tm; i++)
            for (int64_t c = 0; c < tn; c++, f++) {
                if (f < n_full - XS) {
                    if (tile_out) {
                        int32_t *e = tile_out + 4 * nb;
                        e[0] = ORC_TILE; e[1] = s; e[2] = (int32_t)i; e[3] = (int32_t)c;
                    }
                    nb++;
                } else {
                    for (int h = 0; h < 2; h++) {
                        if (tile_out) {
                            int32_t *e = tile_out + 4 * nb;
                            e[0] = ORC_TILE_HALF; e[1] = s; e[2] = (int32_t)i; e[3] = (int32_t)(2 * c + h);
                        }
                        nb++;
                    }
                }
            }
    if (n_transfer) *n_transfer = nt;
    if (n_tile) *n_tile = nb;
    return nt + nb;
}

/* Reduce-scatter rails.
 * Tile rail (one rail for all emulated ranks): TILE(rank q, chunk c, band b,
 * column tile j) = rows [c*m/P + b*R, +R) x columns [j*BN, +BN) of rank q's
 * partial X_q . W_q, written as {2, q*P + c, b, j}.
 *   band order (order = 0): band b outermost, then rank q, then column tile j,
 *     then chunk c [explainer, "Role switching only works": every rank
 *     produces its output band by band across all chunks; the order inside a
 *     band is not given: one rank at a time, column tile outer and chunk
 *     inner keeps the tiles that read one W_q column slice adjacent and one
 *     band of X_q in use, so the operands of the tiles in flight fit in L2;
 *     with all ranks of one GPU interleaved tile by tile they did not];
 *   row order  (order = 1): chunk c, then band b, then rank q, then j (global
 *     row order).
 * Reduce rail of rank r: REDUCE(c = r, band b, column tile j), b outer, j inner.
 * Bands are R rows of a chunk of m/P rows. */
ORC_EXPORT int64_t orc_rail_rs(int P, int64_t m, int64_t n, int R, int BN, int order, int rank,
                               int32_t *tile_out, int64_t *n_tile,
                               int32_t *reduce_out, int64_t *n_reduce) {
    if (m % P) return -1;
    int64_t mc = m / P, bands = orc_cdiv(mc, R), tn = orc_cdiv(n, BN);
    int64_t nb = 0, nr = 0;
    if (order == 0) {
        for (int64_t b = 0; b < bands; b++)
            for (int q = 0; q < P; q++)
                for (int64_t j = 0; j < tn; j++)
                    for (int c = 0; c < P; c++) {
                        if (tile_out) {
                            int32_t *e = tile_out + 4 * nb;
                            e[0] = ORC_TILE; e[1] = q * P + c; e[2] = (int32_t)b; e[3] = (int32_t)j;
                        }
                        nb++;
                    }
    } else {
        for (int c = 0; c < P; c++)
            for (int64_t b = 0; b < bands; b++)
                for (int q = 0; q < P; q++)
                    for (int64_t j = 0; j < tn; j++) {
                        if (tile_out) {
                            int32_t *e = tile_out + 4 * nb;
                            e[0] = ORC_TILE; e[1] = q * P + c; e[2] = (int32_t)b; e[3] = (int32_t)j;
                        }
                        nb++;
                    }
    }
    for (int64_t b = 0; b < bands; b++)
        for (int64_t j = 0; j < tn; j++) {
            if (reduce_out) {
                int32_t *e = reduce_out + 4 * nr;
                e[0] = ORC_REDUCE; e[1] = rank; e[2] = (int32_t)b; e[3] = (int32_t)j;
            }
            nr++;
        }
    if (n_tile) *n_tile = nb;
    if (n_reduce) *n_reduce = nr;
    return nb + nr;
}

/* Number of OpenMP threads the oracle runs with. */
ORC_EXPORT int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
