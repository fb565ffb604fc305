/*
 * Oracle for the gated delta rule layer: plain, slow, fp64, token by token.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests, the smoke check and the benchmark's
 * CPU-baseline leg call this file. The product path (the CUDA library) shares
 * no code, header or constant with it.
 *
 * What it computes (one Qwen3.5-style Gated-DeltaNet layer, per v-head h with
 * q/k head h / (Hv/Hk)):
 *   1. causal short convolution, kernel 4, over each q/k/v channel, with the
 *      last three raw inputs carried as conv state ("The shadow reader",
 *      section "Exact on a grid": the convolution state is part of what a
 *      replay must reproduce; "qwen3_5: run prompts that share prefixes once
 *      per prefix", section "Purpose": a captured state keeps "the last three
 *      conv inputs");
 *   2. L2 normalisation of q and k per head;
 *   3. the gated delta rule S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T)
 *      + beta_t v_t k_t^T with output o_t = S_t q_t.
 * The state is stored transposed, S^T with shape [d_k][d_v], the layout the
 * library's sessions use.
 *
 * Readings where the pages say nothing (each listed in the design notes):
 *   - tap order: w[c][3] multiplies the current token, w[c][0] the token three
 *     positions back (cross-correlation with three positions of left context);
 *   - no conv bias; optional SiLU after the conv (off by default);
 *   - q_hat = q_scale * y / sqrt(|y|^2 + eps), k_hat = y / sqrt(|y|^2 + eps);
 *   - g and beta arrive already activated, one per token and v-head.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (the build step in
 * oracle/build.py). fp contraction is off so x86 and Arm hosts round alike.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

/* Causal conv of one channel block.
 * x: [T][ld_x] values, channels [0, nc) used; w: [nc][4]; state_in/out: [3][nc]
 * (row 0 = oldest). y: [T][nc]. state_out may alias state_in. */
EXPORT void oracle_conv(int64_t T, int64_t nc, const double *x, int64_t ld_x,
                        const double *w, const double *state_in, int act,
                        double *y, double *state_out)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < nc; ++c) {
            double acc = 0.0;
            for (int i = 0; i < 4; ++i) {
                int64_t p = t - 3 + i;                 /* absolute input position of tap i */
                double xv = (p >= 0) ? x[p * ld_x + c] : state_in[(3 + p) * nc + c];
                acc += w[c * 4 + i] * xv;
            }
            if (act == 1) acc = acc / (1.0 + exp(-acc));   /* SiLU */
            y[t * nc + c] = acc;
        }
    }
    /* new conv state: the raw inputs at the last three positions */
    double *tmp = (double *)malloc(sizeof(double) * 3 * (size_t)nc);
    for (int r = 0; r < 3; ++r) {
        int64_t p = T - 3 + r;
        for (int64_t c = 0; c < nc; ++c)
            tmp[r * nc + c] = (p >= 0) ? x[p * ld_x + c] : state_in[(3 + p) * nc + c];
    }
    memcpy(state_out, tmp, sizeof(double) * 3 * (size_t)nc);
    free(tmp);
}

/* Per-head L2 normalisation: out = scale * y / sqrt(sum(y^2) + eps). y, out: [T][H*d]. */
EXPORT void oracle_l2norm(int64_t T, int64_t H, int64_t d, const double *y,
                          double scale, double eps, double *out)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            const double *yy = y + (t * H + h) * d;
            double ss = 0.0;
            for (int64_t i = 0; i < d; ++i) ss += yy[i] * yy[i];
            double r = scale / sqrt(ss + eps);
            for (int64_t i = 0; i < d; ++i) out[(t * H + h) * d + i] = yy[i] * r;
        }
}

/* The recurrence, taking the decay factor alpha_t = exp(g_t) directly.
 * q, k: [T][Hk][dk]; v: [T][Hv][dv]; alpha, beta: [T][Hv];
 * ST: [Hv][dk][dv] in/out (S transposed); o: [T][Hv][dv].
 * Transposed form of the update: S_t^T = alpha (I - beta k k^T) S_{t-1}^T + beta k v^T. */
EXPORT void oracle_recurrence(int64_t T, int Hk, int Hv, int dk, int dv,
                              const double *q, const double *k, const double *v,
                              const double *alpha, const double *beta,
                              double *ST, double *o)
{
    const int G = Hv / Hk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < Hv; ++h) {
        const int hk = h / G;
        double *S = ST + (int64_t)h * dk * dv;
        double *kS = (double *)malloc(sizeof(double) * dv);
        for (int64_t t = 0; t < T; ++t) {
            const double *kt = k + (t * Hk + hk) * dk;
            const double *qt = q + (t * Hk + hk) * dk;
            const double *vt = v + (t * Hv + h) * dv;
            const double a = alpha[t * Hv + h], b = beta[t * Hv + h];
            /* k^T S^T (= (S k)^T), a row over d_v */
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int i = 0; i < dk; ++i) s += kt[i] * S[i * dv + j];
                kS[j] = s;
            }
            /* S^T <- a (S^T - b k (k^T S^T)) + b k v^T */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[i * dv + j] = a * (S[i * dv + j] - b * kt[i] * kS[j]) + b * kt[i] * vt[j];
            /* o_t = S_t q_t, i.e. o_j = sum_i S^T[i][j] q_i */
            double *ot = o + (t * Hv + h) * dv;
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int i = 0; i < dk; ++i) s += S[i * dv + j] * qt[i];
                ot[j] = s;
            }
        }
        free(kS);
    }
}

/* The whole layer over T tokens of one session.
 * xq, xk: [T][Hk*dk]; xv: [T][Hv*dv]; g, beta: [T][Hv];
 * conv_w: [ch][4] with ch = 2*Hk*dk + Hv*dv, channel order q | k | v;
 * conv_state: [3][ch] in/out; ST: [Hv][dk][dv] in/out; o: [T][Hv][dv]. */
EXPORT int oracle_layer(int64_t T, int Hk, int Hv, int dk, int dv, int act,
                        double q_scale, double eps,
                        const double *xq, const double *xk, const double *xv,
                        const double *g, const double *beta, const double *conv_w,
                        double *conv_state, double *ST, double *o)
{
    if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || T < 0) return 1;
    const int64_t nq = (int64_t)Hk * dk, nv = (int64_t)Hv * dv, ch = 2 * nq + nv;
    double *yq = (double *)malloc(sizeof(double) * (size_t)(T * nq + 1));
    double *yk = (double *)malloc(sizeof(double) * (size_t)(T * nq + 1));
    double *yv = (double *)malloc(sizeof(double) * (size_t)(T * nv + 1));
    double *st = (double *)malloc(sizeof(double) * (size_t)(3 * ch));
    double *st_out = (double *)malloc(sizeof(double) * (size_t)(3 * ch));
    double *a = (double *)malloc(sizeof(double) * (size_t)(T * Hv + 1));
    if (!yq || !yk || !yv || !st || !st_out || !a) return 2;

    /* split the conv state into its q, k, v column blocks */
    const double *blocks_x[3] = {xq, xk, xv};
    double *blocks_y[3] = {yq, yk, yv};
    const int64_t off[3] = {0, nq, 2 * nq}, width[3] = {nq, nq, nv};
    for (int b = 0; b < 3; ++b) {
        double *s_in = (double *)malloc(sizeof(double) * 3 * (size_t)width[b]);
        double *s_out = (double *)malloc(sizeof(double) * 3 * (size_t)width[b]);
        double *wb = (double *)malloc(sizeof(double) * 4 * (size_t)width[b]);
        for (int r = 0; r < 3; ++r)
            for (int64_t c = 0; c < width[b]; ++c) s_in[r * width[b] + c] = conv_state[r * ch + off[b] + c];
        for (int64_t c = 0; c < width[b]; ++c)
            for (int i = 0; i < 4; ++i) wb[c * 4 + i] = conv_w[(off[b] + c) * 4 + i];
        oracle_conv(T, width[b], blocks_x[b], width[b], wb, s_in, act, blocks_y[b], s_out);
        for (int r = 0; r < 3; ++r)
            for (int64_t c = 0; c < width[b]; ++c) st_out[r * ch + off[b] + c] = s_out[r * width[b] + c];
        free(s_in); free(s_out); free(wb);
    }
    memcpy(conv_state, st_out, sizeof(double) * 3 * (size_t)ch);

    oracle_l2norm(T, Hk, dk, yq, q_scale, eps, yq);
    oracle_l2norm(T, Hk, dk, yk, 1.0, eps, yk);
    for (int64_t i = 0; i < T * Hv; ++i) a[i] = exp(g[i]);
    oracle_recurrence(T, Hk, Hv, dk, dv, yq, yk, yv, a, beta, ST, o);

    free(yq); free(yk); free(yv); free(st); free(st_out); free(a);
    return 0;
}

/*
 * Gates from raw per-token projections (the optional raw-gate variant). The
 * pages take g and beta as given, already activated; this variant follows the
 * usual Gated-DeltaNet parametrisation of such layers (a reading, not in the
 * pages): per token t and v-head h,
 *   g[t][h]    = -exp(A_log[h]) * softplus(a[t][h] + dt_bias[h]),
 *   beta[t][h] = 1 / (1 + exp(-b[t][h])),
 * with softplus(x) = log(1 + exp(x)), evaluated as max(x, 0) + log1p(exp(-|x|))
 * (the same function, without overflow for large x).
 */
EXPORT void oracle_gates(int64_t T, int Hv, const double *a, const double *b, const double *A_log,
                  const double *dt_bias, double *g, double *beta) {
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < Hv; ++h) {
            const int64_t i = t * Hv + h;
            const double x = a[i] + dt_bias[h];
            const double sp = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
            g[i] = -exp(A_log[h]) * sp;
            beta[i] = 1.0 / (1.0 + exp(-b[i]));
        }
}
