/*
 * CPU oracle for the forward pass of 3-D neighborhood attention (NA3D).
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. It shares no
 * code with the CUDA path: its own index arithmetic, its own bf16 widening,
 * plain fp64 loops in the order the definition states them.
 *
 * What it computes ("[Triton/Gluon] Add 3D neighborhood flash attention
 * (na3d_flash)", ROCm/aiter pull request 5230):
 *   - Motivation: the token at grid position (t,h,w) attends only to its
 *     KT x KH x KW neighbours, not to the whole sequence.
 *   - Technical Details, kernel bullets: windows shift inward at the borders,
 *     so every window holds exactly KT*KH*KW keys.
 *   - Technical Details, launcher: tensors are (B, T, H, W, NH, HD) bf16 and
 *     q arrives already multiplied by head_dim^-0.5, so no scale is applied
 *     here.
 *   - Technical Details, test file: the exact reference is a per-query loop
 *     (there in FP32; here in fp64, from the exactly widened bf16 inputs).
 *
 * Reading of the border shift (the pages say only "inward border-shift,
 * exactly K keys"): on an axis of length N with window length K <= N, the
 * query at i uses keys [s, s + K) with
 *     s = min(max(i - floor(K/2), 0), N - K),
 * the plainest rule that keeps K keys, lies inside [0, N) and centres the
 * window on i away from the borders.
 *
 * For a query p = (b, t, h, w) and head n, with window W(p) (the product of
 * the three axis intervals):
 *     x_j  = sum_d q[p,n,d] * k[j,n,d]                    for j in W(p)
 *     o[d] = sum_j exp(x_j - max x) v[j,n,d] / sum_j exp(x_j - max x)
 * all in fp64.
 *
 * Any 1 <= K <= N is accepted (even K included, which the CUDA path rejects).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: the top 16 bits of an fp32. */
static double bf16_to_f64(uint16_t u) {
    uint32_t b = (uint32_t)u << 16;
    float f;
    memcpy(&f, &b, sizeof f);
    return (double)f;
}

int64_t na3d_oracle_window_start(int64_t i, int64_t K, int64_t N) {
    int64_t s = i - K / 2;
    if (s < 0) s = 0;
    if (s > N - K) s = N - K;
    return s;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int64_t B, T, H, W, NH, HD, KT, KH, KW;
} na3d_problem;

static int check_problem(const na3d_problem* P) {
    if (!P->q || !P->k || !P->v) return 1;
    if (P->B < 1 || P->T < 1 || P->H < 1 || P->W < 1 || P->NH < 1 || P->HD < 1) return 2;
    if (P->KT < 1 || P->KH < 1 || P->KW < 1) return 3;
    if (P->KT > P->T || P->KH > P->H || P->KW > P->W) return 3;
    return 0;
}

/* One query row (b,t,h,w,n). x: scratch of KT*KH*KW doubles, qd: HD doubles.
 * Writes o[0..HD). Optionally reports the window's token indices and the
 * softmax weights (both KT*KH*KW long, in (kt, kh, kw) order). */
static void oracle_query(const na3d_problem* P, int64_t b, int64_t t, int64_t h,
                         int64_t w, int64_t n, double* x, double* qd, double* o,
                         int64_t* key_tokens, double* weights) {
    const int64_t HD = P->HD, NH = P->NH;
    const int64_t tok_q = ((b * P->T + t) * P->H + h) * P->W + w;
    const uint16_t* qrow = P->q + (tok_q * NH + n) * HD;
    for (int64_t d = 0; d < HD; ++d) qd[d] = bf16_to_f64(qrow[d]);

    const int64_t st = na3d_oracle_window_start(t, P->KT, P->T);
    const int64_t sh = na3d_oracle_window_start(h, P->KH, P->H);
    const int64_t sw = na3d_oracle_window_start(w, P->KW, P->W);

    /* scores over the explicit window */
    int64_t j = 0;
    double xmax = -INFINITY;
    for (int64_t kt = st; kt < st + P->KT; ++kt)
        for (int64_t kh = sh; kh < sh + P->KH; ++kh)
            for (int64_t kw = sw; kw < sw + P->KW; ++kw, ++j) {
                const int64_t tok = ((b * P->T + kt) * P->H + kh) * P->W + kw;
                const uint16_t* krow = P->k + (tok * NH + n) * HD;
                double acc = 0.0;
                for (int64_t d = 0; d < HD; ++d) acc += qd[d] * bf16_to_f64(krow[d]);
                x[j] = acc;
                if (acc > xmax) xmax = acc;
                if (key_tokens) key_tokens[j] = tok;
            }

    /* softmax over the window, then the weighted sum of v */
    double denom = 0.0;
    for (int64_t i = 0; i < j; ++i) {
        x[i] = exp(x[i] - xmax);
        denom += x[i];
    }
    for (int64_t d = 0; d < HD; ++d) o[d] = 0.0;
    j = 0;
    for (int64_t kt = st; kt < st + P->KT; ++kt)
        for (int64_t kh = sh; kh < sh + P->KH; ++kh)
            for (int64_t kw = sw; kw < sw + P->KW; ++kw, ++j) {
                const int64_t tok = ((b * P->T + kt) * P->H + kh) * P->W + kw;
                const uint16_t* vrow = P->v + (tok * NH + n) * HD;
                const double wgt = x[j] / denom;
                if (weights) weights[j] = wgt;
                for (int64_t d = 0; d < HD; ++d) o[d] += wgt * bf16_to_f64(vrow[d]);
            }
}

/* Decompose a flat row index over (B, T, H, W, NH). */
static void split_row(const na3d_problem* P, int64_t row, int64_t* b, int64_t* t,
                      int64_t* h, int64_t* w, int64_t* n) {
    *n = row % P->NH; row /= P->NH;
    *w = row % P->W;  row /= P->W;
    *h = row % P->H;  row /= P->H;
    *t = row % P->T;  row /= P->T;
    *b = row;
}

/* Output rows `rows[0..n_rows)` (flat indices over (B,T,H,W,NH)) into
 * out[i*HD .. (i+1)*HD). Returns 0, or a nonzero code for invalid arguments. */
int na3d_oracle_fwd_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int64_t* rows, int64_t n_rows, double* out,
                         int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH,
                         int64_t HD, int64_t KT, int64_t KH, int64_t KW, int nthreads) {
    na3d_problem P = {q, k, v, B, T, H, W, NH, HD, KT, KH, KW};
    int err = check_problem(&P);
    if (err) return err;
    if (!out || (n_rows > 0 && !rows)) return 1;
    const int64_t total = B * T * H * W * NH;
    for (int64_t i = 0; i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total) return 4;
    const int64_t KK = KT * KH * KW;
    int fail = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt) reduction(| : fail)
#endif
    {
        double* x = (double*)malloc((size_t)KK * sizeof(double));
        double* qd = (double*)malloc((size_t)HD * sizeof(double));
        if (!x || !qd) {
            fail = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 64)
#endif
            for (int64_t i = 0; i < n_rows; ++i) {
                int64_t b, t, h, w, n;
                split_row(&P, rows[i], &b, &t, &h, &w, &n);
                oracle_query(&P, b, t, h, w, n, x, qd, out + i * HD, NULL, NULL);
            }
        }
        free(x);
        free(qd);
    }
    return fail ? 5 : 0;
}

/* The whole output tensor, fp64, same (B,T,H,W,NH,HD) layout as the inputs. */
int na3d_oracle_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, double* out,
                    int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD,
                    int64_t KT, int64_t KH, int64_t KW, int nthreads) {
    na3d_problem P = {q, k, v, B, T, H, W, NH, HD, KT, KH, KW};
    int err = check_problem(&P);
    if (err) return err;
    if (!out) return 1;
    const int64_t total = B * T * H * W * NH;
    const int64_t KK = KT * KH * KW;
    int fail = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt) reduction(| : fail)
#endif
    {
        double* x = (double*)malloc((size_t)KK * sizeof(double));
        double* qd = (double*)malloc((size_t)HD * sizeof(double));
        if (!x || !qd) {
            fail = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 64)
#endif
            for (int64_t row = 0; row < total; ++row) {
                int64_t b, t, h, w, n;
                split_row(&P, row, &b, &t, &h, &w, &n);
                oracle_query(&P, b, t, h, w, n, x, qd, out + row * HD, NULL, NULL);
            }
        }
        free(x);
        free(qd);
    }
    return fail ? 5 : 0;
}

/* One row with its internals: the KT*KH*KW window token indices (flat over
 * (B,T,H,W)), the softmax weights, and the output row. */
int na3d_oracle_row_detail(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           int64_t row, int64_t* key_tokens, double* weights, double* o,
                           int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH,
                           int64_t HD, int64_t KT, int64_t KH, int64_t KW) {
    na3d_problem P = {q, k, v, B, T, H, W, NH, HD, KT, KH, KW};
    int err = check_problem(&P);
    if (err) return err;
    if (!key_tokens || !weights || !o) return 1;
    if (row < 0 || row >= B * T * H * W * NH) return 4;
    const int64_t KK = KT * KH * KW;
    double* x = (double*)malloc((size_t)KK * sizeof(double));
    double* qd = (double*)malloc((size_t)HD * sizeof(double));
    if (!x || !qd) {
        free(x);
        free(qd);
        return 5;
    }
    int64_t b, t, h, w, n;
    split_row(&P, row, &b, &t, &h, &w, &n);
    oracle_query(&P, b, t, h, w, n, x, qd, o, key_tokens, weights);
    free(x);
    free(qd);
    return 0;
}
