/*
 * gma_oracle.c -- fp64 CPU oracle for the Gaussian Mixture Attention (GMA) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file exists so that the tests, the smoke check and the
 * benchmark's CPU-baseline leg can compare the CUDA library against a plain, slow, obviously
 * correct statement of what GMA computes.  No product code path links, loads or calls it, and it
 * shares no code, header, table or helper with the CUDA library.
 *
 * Source of the definitions: "Résumé Technique : Attention par Mélange Gaussien (GMA)"
 * (gist.science/fr/paper/2606.18283), section "Méthodologie", subsections
 *   1. "Routage Latent Probabiliste"            -- the GMM posterior responsibilities,
 *   2. "Routage de Mémoire Latente"             -- write phase, read phase and the displayed
 *                                                  equation O = Gamma_Q V~ / (Gamma_Q Z + eps),
 *   3. "Variantes et Entraînement"              -- causal variant by prefix sums; softplus
 *                                                  variances and softmax priors.
 *
 * Everything is computed in double precision, one token at a time, in the order the page
 * states the steps.  Readings taken where the page is silent:
 *   - one GMM per head, shared by queries and keys ("espace latent partagé");
 *   - sigma^2 = softplus(raw) + var_floor, with softplus(r) = log(1 + e^r) evaluated stably;
 *   - pi = softmax(prior logits);
 *   - the Gaussian log-density includes the log-determinant term; the -d/2 log(2 pi) constant is
 *     the same for every component and cancels in the posterior, so it is left out;
 *   - eps is a scalar added to each query row's normaliser;
 *   - the causal prefix is inclusive (token i sees keys j <= i).
 *
 * Layouts (row-major, contiguous): activations [B][H][N][d], parameters mu and raw [H][K][d_r],
 * prior logits [H][K], output O [B][H][N][d_v].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(r) = log(1 + exp(r)), written so that it neither overflows for large r nor loses
 * the small tail for very negative r. */
static double oracle_softplus(double r)
{
    return (r > 0.0 ? r : 0.0) + log1p(exp(-fabs(r)));
}

/* Reparametrisation ("softplus pour les variances, softmax pour les prioris"):
 *   var[k][d]  = softplus(raw[k][d]) + var_floor
 *   logpi[k]   = logits[k] - log sum_k' exp(logits[k'])
 */
void gmao_params(int K, int d_r, const double *raw, const double *logits, double var_floor,
                 double *var, double *logpi)
{
    for (int i = 0; i < K * d_r; ++i)
        var[i] = oracle_softplus(raw[i]) + var_floor;
    double m = -INFINITY;
    for (int k = 0; k < K; ++k)
        if (logits[k] > m) m = logits[k];
    double s = 0.0;
    for (int k = 0; k < K; ++k)
        s += exp(logits[k] - m);
    double lse = m + log(s);
    for (int k = 0; k < K; ++k)
        logpi[k] = logits[k] - lse;
}

/* Posterior responsibility of one routing vector x (length d_r) over K diagonal Gaussians:
 *   L_k     = log pi_k - 1/2 sum_d [ (x_d - mu_kd)^2 / var_kd + log var_kd ]
 *   gamma_k = exp(L_k - max L) / sum_k' exp(L_k' - max L)          ( = p(z = k | x) )
 * `work` holds K doubles of scratch. */
static void oracle_posterior(int d_r, int K, const double *x, const double *mu, const double *var,
                             const double *logpi, double *gamma, double *work)
{
    double mx = -INFINITY;
    for (int k = 0; k < K; ++k) {
        double q = 0.0;
        const double *mk = mu + (size_t)k * d_r;
        const double *vk = var + (size_t)k * d_r;
        for (int d = 0; d < d_r; ++d) {
            double diff = x[d] - mk[d];
            q += diff * diff / vk[d] + log(vk[d]);
        }
        work[k] = logpi[k] - 0.5 * q;
        if (work[k] > mx) mx = work[k];
    }
    double s = 0.0;
    for (int k = 0; k < K; ++k) {
        gamma[k] = exp(work[k] - mx);
        s += gamma[k];
    }
    for (int k = 0; k < K; ++k)
        gamma[k] /= s;
}

/* Responsibilities of N routing vectors X [N][d_r] for one head: gamma [N][K]. */
void gmao_responsibilities(int N, int d_r, int K, const double *X, const double *mu,
                           const double *raw, const double *logits, double var_floor,
                           double *gamma)
{
    double *var = (double *)malloc(sizeof(double) * (size_t)K * d_r);
    double *logpi = (double *)malloc(sizeof(double) * (size_t)K);
    double *work = (double *)malloc(sizeof(double) * (size_t)K);
    gmao_params(K, d_r, raw, logits, var_floor, var, logpi);
    for (int i = 0; i < N; ++i)
        oracle_posterior(d_r, K, X + (size_t)i * d_r, mu, var, logpi, gamma + (size_t)i * K, work);
    free(var);
    free(logpi);
    free(work);
}

/* One (batch, head) slice of the forward pass.
 *
 * Bidirectional (write phase, then read phase):
 *   Vt[k][:] = sum_j gamma_K[j][k] v_j          (latent memory  V~ = Gamma_K^T V)
 *   Z[k]     = sum_j gamma_K[j][k]              (normaliser     Z  = Gamma_K^T 1)
 *   O_i      = (gamma_Q[i] . Vt) / (gamma_Q[i] . Z + eps)
 *
 * Causal (prefix sums of the memory and the normaliser, inclusive of j = i):
 *   for i = 0 .. N-1:  Vt += gamma_K[i] v_i^T;  Z += gamma_K[i];
 *                      O_i = (gamma_Q[i] . Vt) / (gamma_Q[i] . Z + eps)
 */
static void oracle_slice(int causal, int N, int d_r, int K, int d_v, const double *QX,
                         const double *KX, const double *V, const double *mu, const double *var,
                         const double *logpi, double eps, double *O)
{
    double *Vt = (double *)calloc((size_t)K * d_v, sizeof(double));
    double *Z = (double *)calloc((size_t)K, sizeof(double));
    double *gk = (double *)malloc(sizeof(double) * (size_t)K);
    double *gq = (double *)malloc(sizeof(double) * (size_t)K);
    double *work = (double *)malloc(sizeof(double) * (size_t)K);
    double *num = (double *)malloc(sizeof(double) * (size_t)d_v);

    if (!causal) {
        for (int j = 0; j < N; ++j) {
            oracle_posterior(d_r, K, KX + (size_t)j * d_r, mu, var, logpi, gk, work);
            const double *vj = V + (size_t)j * d_v;
            for (int k = 0; k < K; ++k) {
                Z[k] += gk[k];
                double *row = Vt + (size_t)k * d_v;
                for (int c = 0; c < d_v; ++c)
                    row[c] += gk[k] * vj[c];
            }
        }
    }
    for (int i = 0; i < N; ++i) {
        if (causal) {
            oracle_posterior(d_r, K, KX + (size_t)i * d_r, mu, var, logpi, gk, work);
            const double *vi = V + (size_t)i * d_v;
            for (int k = 0; k < K; ++k) {
                Z[k] += gk[k];
                double *row = Vt + (size_t)k * d_v;
                for (int c = 0; c < d_v; ++c)
                    row[c] += gk[k] * vi[c];
            }
        }
        oracle_posterior(d_r, K, QX + (size_t)i * d_r, mu, var, logpi, gq, work);
        double den = 0.0;
        for (int c = 0; c < d_v; ++c)
            num[c] = 0.0;
        for (int k = 0; k < K; ++k) {
            den += gq[k] * Z[k];
            const double *row = Vt + (size_t)k * d_v;
            for (int c = 0; c < d_v; ++c)
                num[c] += gq[k] * row[c];
        }
        double *oi = O + (size_t)i * d_v;
        for (int c = 0; c < d_v; ++c)
            oi[c] = num[c] / (den + eps);
    }
    free(Vt);
    free(Z);
    free(gk);
    free(gq);
    free(work);
    free(num);
}

/* Full forward pass over B x H slices.  Parameters are per head and shared across the batch.
 * nthreads <= 0 lets OpenMP choose.  Returns the number of threads used. */
int gmao_forward(int causal, int B, int H, int N, int d_r, int K, int d_v, const double *QX,
                 const double *KX, const double *V, const double *mu, const double *raw,
                 const double *logits, double var_floor, double eps, double *O, int nthreads)
{
    double *var = (double *)malloc(sizeof(double) * (size_t)H * K * d_r);
    double *logpi = (double *)malloc(sizeof(double) * (size_t)H * K);
    for (int h = 0; h < H; ++h)
        gmao_params(K, d_r, raw + (size_t)h * K * d_r, logits + (size_t)h * K, var_floor,
                    var + (size_t)h * K * d_r, logpi + (size_t)h * K);
    int used = 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
    {
#pragma omp single
        used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 1)
        for (int bh = 0; bh < B * H; ++bh) {
#else
    (void)nthreads;
    {
        for (int bh = 0; bh < B * H; ++bh) {
#endif
            int h = bh % H;
            size_t s = (size_t)bh * N;
            oracle_slice(causal, N, d_r, K, d_v, QX + s * d_r, KX + s * d_r, V + s * d_v,
                         mu + (size_t)h * K * d_r, var + (size_t)h * K * d_r,
                         logpi + (size_t)h * K, eps, O + s * d_v);
        }
    }
    free(var);
    free(logpi);
    return used;
}

/* One autoregressive decode step per (batch, head) slice: the causal variant (Méthodologie §3) for
 * one new token whose key and value join the prefix before its query reads it.
 *   gamma_K = p(z | kx);   S[k][c] += gamma_K[k] v[c]  (c < d_v);   S[k][d_v] += gamma_K[k]
 *   gamma_Q = p(z | qx);   o[c] = (gamma_Q . S[:, c]) / (gamma_Q . S[:, d_v] + eps)
 * qx, kx [B][H][d_r]; v [B][H][d_v]; state [B][H][K][d_v + 1], updated in place; o [B][H][d_v]. */
void gmao_decode_step(int B, int H, int d_r, int K, int d_v, const double *qx, const double *kx,
                      const double *v, const double *mu, const double *raw, const double *logits,
                      double var_floor, double eps, double *state, double *o)
{
    double *var = (double *)malloc(sizeof(double) * (size_t)K * d_r);
    double *logpi = (double *)malloc(sizeof(double) * (size_t)K);
    double *gk = (double *)malloc(sizeof(double) * (size_t)K);
    double *gq = (double *)malloc(sizeof(double) * (size_t)K);
    double *work = (double *)malloc(sizeof(double) * (size_t)K);
    const int ne = d_v + 1;
    for (int bh = 0; bh < B * H; ++bh) {
        const int h = bh % H;
        gmao_params(K, d_r, raw + (size_t)h * K * d_r, logits + (size_t)h * K, var_floor, var, logpi);
        const double *muh = mu + (size_t)h * K * d_r;
        oracle_posterior(d_r, K, kx + (size_t)bh * d_r, muh, var, logpi, gk, work);
        oracle_posterior(d_r, K, qx + (size_t)bh * d_r, muh, var, logpi, gq, work);
        double *S = state + (size_t)bh * K * ne;
        const double *vb = v + (size_t)bh * d_v;
        for (int k = 0; k < K; ++k) {
            for (int c = 0; c < d_v; ++c)
                S[(size_t)k * ne + c] += gk[k] * vb[c];
            S[(size_t)k * ne + d_v] += gk[k];
        }
        double den = 0.0;
        for (int k = 0; k < K; ++k)
            den += gq[k] * S[(size_t)k * ne + d_v];
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k)
                num += gq[k] * S[(size_t)k * ne + c];
            o[(size_t)bh * d_v + c] = num / (den + eps);
        }
    }
    free(var);
    free(logpi);
    free(gk);
    free(gq);
    free(work);
}

/* Cross-attention on the bidirectional path: the Nk keys and values of a slice write the memory
 * (Méthodologie §2, write phase) and the Nq queries read it (read phase).
 * QX [B][H][Nq][d_r]; KX [B][H][Nk][d_r]; V [B][H][Nk][d_v]; O [B][H][Nq][d_v]. */
int gmao_forward_cross(int B, int H, int Nq, int Nk, int d_r, int K, int d_v, const double *QX,
                       const double *KX, const double *V, const double *mu, const double *raw,
                       const double *logits, double var_floor, double eps, double *O)
{
    double *var = (double *)malloc(sizeof(double) * (size_t)K * d_r);
    double *logpi = (double *)malloc(sizeof(double) * (size_t)K);
    double *Vt = (double *)malloc(sizeof(double) * (size_t)K * d_v);
    double *Z = (double *)malloc(sizeof(double) * (size_t)K);
    double *g = (double *)malloc(sizeof(double) * (size_t)K);
    double *work = (double *)malloc(sizeof(double) * (size_t)K);
    for (int bh = 0; bh < B * H; ++bh) {
        const int h = bh % H;
        gmao_params(K, d_r, raw + (size_t)h * K * d_r, logits + (size_t)h * K, var_floor, var, logpi);
        const double *muh = mu + (size_t)h * K * d_r;
        for (int i = 0; i < K * d_v; ++i)
            Vt[i] = 0.0;
        for (int k = 0; k < K; ++k)
            Z[k] = 0.0;
        for (int j = 0; j < Nk; ++j) {
            oracle_posterior(d_r, K, KX + ((size_t)bh * Nk + j) * d_r, muh, var, logpi, g, work);
            const double *vj = V + ((size_t)bh * Nk + j) * d_v;
            for (int k = 0; k < K; ++k) {
                Z[k] += g[k];
                for (int c = 0; c < d_v; ++c)
                    Vt[(size_t)k * d_v + c] += g[k] * vj[c];
            }
        }
        for (int i = 0; i < Nq; ++i) {
            oracle_posterior(d_r, K, QX + ((size_t)bh * Nq + i) * d_r, muh, var, logpi, g, work);
            double den = 0.0;
            for (int k = 0; k < K; ++k)
                den += g[k] * Z[k];
            double *oi = O + ((size_t)bh * Nq + i) * d_v;
            for (int c = 0; c < d_v; ++c) {
                double num = 0.0;
                for (int k = 0; k < K; ++k)
                    num += g[k] * Vt[(size_t)k * d_v + c];
                oi[c] = num / (den + eps);
            }
        }
    }
    free(var);
    free(logpi);
    free(Vt);
    free(Z);
    free(g);
    free(work);
    return 1;
}

