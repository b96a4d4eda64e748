/*
 * Plain fp64 CPU oracle for the Gaussian Mixture Attention (GMA) forward, its
 * cross-attention and diagnostics variants, and its backward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library shares no
 * code with it and never calls it.
 *
 * Source: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 * Probabilistic Latent Routing" (Huang & Raza, 2026), sections 3-5.  Every
 * function below evaluates the paper's definitions directly, in double
 * precision, in the order the equations are written:
 *
 *   Eq. (14)  sigma^2_{k,m} = log(1 + exp(omega_{k,m})) + eps_sigma
 *   Eq. (15)  pi_k = softmax(alpha)_k              (used as log pi_k)
 *   Eq. (16)  s_{i,k} = log pi_k - (d/2) log(2 pi) - (1/2) log|Sigma_k|
 *                       - (1/2) (x_i - mu_k)^T Sigma_k^{-1} (x_i - mu_k)
 *   Eq. (3b)  gamma_{i,k} = exp(s_{i,k}) / sum_l exp(s_{i,l})
 *   Eq. (5-6) Vt_k = sum_j gamma^K_{j,k} V_j,  Z_k = sum_j gamma^K_{j,k}
 *   Eq. (7-8) O_i = sum_k gamma^Q_{i,k} Vt_k / (sum_k gamma^Q_{i,k} Z_k + eps)
 *   Eq. (6b)  causal prefix memory: sums over j <= i (inclusive)
 *   Eq. (8b)  causal read from the prefix memory of position i
 *   Eq. (24)-(29)  responsibility diagnostics (section 5.4)
 *   Eq. (17)-(20)  backward pass (section 4.1; see gma_oracle_backward_head)
 *
 * Readings where the paper leaves a step open:
 *   - softplus is evaluated as max(w,0) + log1p(exp(-|w|)), which equals
 *     log(1+exp(w)) exactly in real arithmetic and does not overflow;
 *   - the softmax subtracts the row maximum before exponentiating (the
 *     paper fixes the value, not the evaluation order);
 *   - the causal prefix is inclusive (row i reads its own key), following
 *     the j <= i of Eq. (6b);
 *   - eps is added once to the scalar denominator of each row (Eq. 8/8b).
 *
 * Layouts: row-major.  X [N, d], V [N, dv], out [N, dv] per head;
 * mu, omega [K, d], alpha [K] per head.  Multi-head drivers take
 * Qx, Kx [G, N, d], V [G, N, dv], out [G, N, dv] with G = B*H heads, and
 * parameters [H, K, d] / [H, K] shared across the batch (head g uses
 * parameter set g % H).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define GMA_ORACLE_LOG_2PI 1.8378770664093454835606594728112

/* Eq. (14): diagonal variance from its unconstrained parameter. */
static double variance_from_omega(double w, double var_floor)
{
    double softplus = (w > 0.0 ? w : 0.0) + log1p(exp(-fabs(w)));
    return softplus + var_floor;
}

/* Eq. (15): log of the softmax-normalised mixture priors. */
static void log_priors(int K, const double *alpha, double *logpi)
{
    double m = alpha[0];
    for (int k = 1; k < K; ++k)
        if (alpha[k] > m) m = alpha[k];
    double sum = 0.0;
    for (int k = 0; k < K; ++k) sum += exp(alpha[k] - m);
    double lse = m + log(sum);
    for (int k = 0; k < K; ++k) logpi[k] = alpha[k] - lse;
}

/*
 * Eq. (16): pre-normalised log-density scores s [N, K] of the rows of X.
 * Direct Mahalanobis form, one (i, k) pair at a time.
 */
int gma_oracle_scores(int N, int d, int K, const double *X, const double *mu,
                      const double *omega, const double *alpha, double var_floor,
                      double *s)
{
    if (N < 0 || d <= 0 || K <= 0) return 1;
    double *logpi = (double *)malloc(sizeof(double) * K);
    double *var = (double *)malloc(sizeof(double) * (size_t)K * d);
    if (!logpi || !var) { free(logpi); free(var); return 2; }
    log_priors(K, alpha, logpi);
    for (int k = 0; k < K; ++k)
        for (int m = 0; m < d; ++m)
            var[(size_t)k * d + m] = variance_from_omega(omega[(size_t)k * d + m], var_floor);
    for (int i = 0; i < N; ++i) {
        const double *x = X + (size_t)i * d;
        for (int k = 0; k < K; ++k) {
            const double *mk = mu + (size_t)k * d;
            const double *vk = var + (size_t)k * d;
            double logdet = 0.0, maha = 0.0;
            for (int m = 0; m < d; ++m) {
                double diff = x[m] - mk[m];
                logdet += log(vk[m]);
                maha += diff * diff / vk[m];
            }
            s[(size_t)i * K + k] = logpi[k] - 0.5 * d * GMA_ORACLE_LOG_2PI - 0.5 * logdet - 0.5 * maha;
        }
    }
    free(logpi);
    free(var);
    return 0;
}

/* Eq. (3b): responsibilities gamma [N, K], each row a softmax of its scores. */
int gma_oracle_responsibilities(int N, int d, int K, const double *X, const double *mu,
                                const double *omega, const double *alpha, double var_floor,
                                double *gamma)
{
    int rc = gma_oracle_scores(N, d, K, X, mu, omega, alpha, var_floor, gamma);
    if (rc) return rc;
    for (int i = 0; i < N; ++i) {
        double *row = gamma + (size_t)i * K;
        double m = row[0];
        for (int k = 1; k < K; ++k)
            if (row[k] > m) m = row[k];
        double sum = 0.0;
        for (int k = 0; k < K; ++k) {
            row[k] = exp(row[k] - m);
            sum += row[k];
        }
        for (int k = 0; k < K; ++k) row[k] /= sum;
    }
    return 0;
}

/*
 * One head of the forward.  causal = 0: Eq. (5)-(8).  causal = 1: Eq. (6b),
 * (8b), evaluated as one pass over positions that first adds position i to
 * the prefix memory and then reads it.
 * Optional outputs (may be NULL): Vt [K, dv] and Z [K] -- the full-sequence
 * memory (bidirectional) or the memory after the last position (causal).
 */
int gma_oracle_forward_head(int N, int d, int K, int dv, const double *Qx, const double *Kx,
                            const double *V, const double *mu, const double *omega,
                            const double *alpha, double var_floor, double eps, int causal,
                            double *out, double *Vt_out, double *Z_out)
{
    if (N < 0 || d <= 0 || K <= 0 || dv <= 0) return 1;
    size_t nk = (size_t)N * K;
    double *gq = (double *)malloc(sizeof(double) * (nk ? nk : 1));
    double *gk = (double *)malloc(sizeof(double) * (nk ? nk : 1));
    double *Vt = (double *)calloc((size_t)K * dv, sizeof(double));
    double *Z = (double *)calloc((size_t)K, sizeof(double));
    int rc = 2;
    if (!gq || !gk || !Vt || !Z) goto done;
    rc = gma_oracle_responsibilities(N, d, K, Qx, mu, omega, alpha, var_floor, gq);
    if (rc) goto done;
    rc = gma_oracle_responsibilities(N, d, K, Kx, mu, omega, alpha, var_floor, gk);
    if (rc) goto done;

    if (!causal) {
        /* Eq. (5)-(6): latent memory and normaliser over the whole sequence. */
        for (int j = 0; j < N; ++j)
            for (int k = 0; k < K; ++k) {
                double g = gk[(size_t)j * K + k];
                Z[k] += g;
                for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g * V[(size_t)j * dv + c];
            }
        /* Eq. (7)-(8): normalised read. */
        for (int i = 0; i < N; ++i) {
            double den = 0.0;
            for (int k = 0; k < K; ++k) den += gq[(size_t)i * K + k] * Z[k];
            den += eps;
            for (int c = 0; c < dv; ++c) {
                double num = 0.0;
                for (int k = 0; k < K; ++k) num += gq[(size_t)i * K + k] * Vt[(size_t)k * dv + c];
                out[(size_t)i * dv + c] = num / den;
            }
        }
    } else {
        /* Eq. (6b), (8b): prefix memory including position i, then the read. */
        for (int i = 0; i < N; ++i) {
            for (int k = 0; k < K; ++k) {
                double g = gk[(size_t)i * K + k];
                Z[k] += g;
                for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g * V[(size_t)i * dv + c];
            }
            double den = 0.0;
            for (int k = 0; k < K; ++k) den += gq[(size_t)i * K + k] * Z[k];
            den += eps;
            for (int c = 0; c < dv; ++c) {
                double num = 0.0;
                for (int k = 0; k < K; ++k) num += gq[(size_t)i * K + k] * Vt[(size_t)k * dv + c];
                out[(size_t)i * dv + c] = num / den;
            }
        }
    }
    if (Vt_out) memcpy(Vt_out, Vt, sizeof(double) * (size_t)K * dv);
    if (Z_out) memcpy(Z_out, Z, sizeof(double) * (size_t)K);
    rc = 0;
done:
    free(gq);
    free(gk);
    free(Vt);
    free(Z);
    return rc;
}

/* ---- multi-head driver: heads are independent; one POSIX thread per stripe ---- */

typedef struct {
    int G, H, N, d, K, dv, causal, first, stride;
    const double *Qx, *Kx, *V, *mu, *omega, *alpha;
    double var_floor, eps;
    double *out;
    int rc;
} oracle_job;

static void *oracle_worker(void *arg)
{
    oracle_job *j = (oracle_job *)arg;
    j->rc = 0;
    for (int g = j->first; g < j->G; g += j->stride) {
        int h = g % j->H;
        int rc = gma_oracle_forward_head(
            j->N, j->d, j->K, j->dv, j->Qx + (size_t)g * j->N * j->d,
            j->Kx + (size_t)g * j->N * j->d, j->V + (size_t)g * j->N * j->dv,
            j->mu + (size_t)h * j->K * j->d, j->omega + (size_t)h * j->K * j->d,
            j->alpha + (size_t)h * j->K, j->var_floor, j->eps, j->causal,
            j->out + (size_t)g * j->N * j->dv, NULL, NULL);
        if (rc) j->rc = rc;
    }
    return NULL;
}

/*
 * All G = B*H heads.  threads <= 0 means one thread.  Returns 0 on success.
 */
int gma_oracle_forward(int B, int H, int N, int d, int K, int dv, const double *Qx,
                       const double *Kx, const double *V, const double *mu, const double *omega,
                       const double *alpha, double var_floor, double eps, int causal,
                       double *out, int threads)
{
    if (B <= 0 || H <= 0) return 1;
    int G = B * H;
    if (threads <= 0) threads = 1;
    if (threads > G) threads = G;
    oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return 2; }
    for (int t = 0; t < threads; ++t) {
        oracle_job j = {G, H, N, d, K, dv, causal, t, threads, Qx, Kx, V, mu, omega, alpha,
                        var_floor, eps, out, 0};
        jobs[t] = j;
    }
    int rc = 0;
    for (int t = 1; t < threads; ++t)
        if (pthread_create(&tid[t], NULL, oracle_worker, &jobs[t])) { jobs[t].rc = 3; tid[t] = 0; }
    oracle_worker(&jobs[0]);
    for (int t = 1; t < threads; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    for (int t = 0; t < threads; ++t)
        if (jobs[t].rc) rc = jobs[t].rc;
    free(jobs);
    free(tid);
    return rc;
}

/*
 * Responsibility diagnostics ("Gaussian Mixture Attention", section 5.4,
 * Eqs. 24-29), on the query responsibilities of every head:
 *
 *   Eq. (24)  gbar_{t,k} = (1/H) sum_h gamma^Q_{t,h,k}    (t = (b, position): one token)
 *   Eq. (25)  p_k        = (1/T) sum_t gbar_{t,k}          (T = B N tokens)
 *   Eq. (26)  H_usage    = -sum_k p_k log p_k / log K
 *   Eq. (27)  H_token    = (1/T) sum_t [ -sum_k gbar_{t,k} log gbar_{t,k} ] / log K
 *   Eq. (28)  R_max      = (1/T) sum_t max_k gbar_{t,k}
 *   Eq. (29)  z_t        = argmax_k gbar_{t,k}
 *
 * Readings: 0 log 0 = 0 (the limit); an argmax tie goes to the lowest index;
 * K >= 2 (the normalisation by log K).  Qx [B, H, N, d] (head g = b H + h uses
 * parameter set h).  Outputs: p [K], stats = {H_usage, H_token, R_max}, z [B N]
 * (may be NULL).
 */
int gma_oracle_diagnostics(int B, int H, int N, int d, int K, const double *Qx, const double *mu,
                           const double *omega, const double *alpha, double var_floor, double *p,
                           double *stats, int *z)
{
    if (B <= 0 || H <= 0 || N < 0 || K < 2) return 1;
    double *gam = (double *)malloc(sizeof(double) * (size_t)H * N * K);     /* one batch entry, all heads */
    double *gbar = (double *)malloc(sizeof(double) * (size_t)K);
    if (!gam || !gbar) { free(gam); free(gbar); return 2; }
    for (int k = 0; k < K; ++k) p[k] = 0.0;
    double htok = 0.0, rmax = 0.0;
    const double T = (double)B * (double)N;
    int rc = 0;
    for (int b = 0; b < B && !rc; ++b) {
        for (int h = 0; h < H && !rc; ++h)
            rc = gma_oracle_responsibilities(N, d, K, Qx + ((size_t)b * H + h) * N * d,
                                             mu + (size_t)h * K * d, omega + (size_t)h * K * d,
                                             alpha + (size_t)h * K, var_floor, gam + (size_t)h * N * K);
        for (int i = 0; i < N && !rc; ++i) {
            /* Eq. (24) */
            for (int k = 0; k < K; ++k) {
                double s = 0.0;
                for (int h = 0; h < H; ++h) s += gam[((size_t)h * N + i) * K + k];
                gbar[k] = s / H;
            }
            double ent = 0.0, mx = gbar[0];
            int arg = 0;
            for (int k = 0; k < K; ++k) {
                p[k] += gbar[k];                                            /* Eq. (25), summed */
                if (gbar[k] > 0.0) ent -= gbar[k] * log(gbar[k]);           /* Eq. (27) term */
                if (gbar[k] > mx) { mx = gbar[k]; arg = k; }                /* Eq. (28), (29) */
            }
            htok += ent;
            rmax += mx;
            if (z) z[(size_t)b * N + i] = arg;
        }
    }
    if (!rc) {
        double husage = 0.0;
        for (int k = 0; k < K; ++k) {
            p[k] /= T;
            if (p[k] > 0.0) husage -= p[k] * log(p[k]);                     /* Eq. (26) */
        }
        stats[0] = husage / log((double)K);
        stats[1] = htok / T / log((double)K);
        stats[2] = rmax / T;
    }
    free(gam);
    free(gbar);
    return rc;
}

/*
 * Cross-attention GMA, one head ("Gaussian Mixture Attention", section 3.1 and
 * section 6): queries from a query-side sequence X (Nq rows), keys and values
 * from a context sequence Y (Nkv rows), responsibilities Gamma^Q_X and
 * Gamma^K_Y under the head's one mixture; then Eq. (5)-(8) with the context's
 * memory: Vt = Gamma^K_Y^T V_Y, Z = Gamma^K_Y^T 1, O = Gamma^Q_X Vt / (Gamma^Q_X Z + eps).
 * Bidirectional only (no causal order exists between two sequences).
 * Qx [Nq, d], Ky [Nkv, d], Vy [Nkv, dv] -> out [Nq, dv].
 */
int gma_oracle_cross_head(int Nq, int Nkv, int d, int K, int dv, const double *Qx, const double *Ky,
                          const double *Vy, const double *mu, const double *omega, const double *alpha,
                          double var_floor, double eps, double *out)
{
    if (Nq < 0 || Nkv < 0 || d <= 0 || K <= 0 || dv <= 0) return 1;
    double *gq = (double *)malloc(sizeof(double) * ((size_t)Nq * K + 1));
    double *gk = (double *)malloc(sizeof(double) * ((size_t)Nkv * K + 1));
    double *Vt = (double *)calloc((size_t)K * dv, sizeof(double));
    double *Z = (double *)calloc((size_t)K, sizeof(double));
    int rc = 2;
    if (!gq || !gk || !Vt || !Z) goto done;
    rc = gma_oracle_responsibilities(Nq, d, K, Qx, mu, omega, alpha, var_floor, gq);
    if (rc) goto done;
    rc = gma_oracle_responsibilities(Nkv, d, K, Ky, mu, omega, alpha, var_floor, gk);
    if (rc) goto done;
    /* Eq. (5)-(6) over the context */
    for (int j = 0; j < Nkv; ++j)
        for (int k = 0; k < K; ++k) {
            double g = gk[(size_t)j * K + k];
            Z[k] += g;
            for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g * Vy[(size_t)j * dv + c];
        }
    /* Eq. (7)-(8) for the queries */
    for (int i = 0; i < Nq; ++i) {
        double den = 0.0;
        for (int k = 0; k < K; ++k) den += gq[(size_t)i * K + k] * Z[k];
        den += eps;
        for (int c = 0; c < dv; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gq[(size_t)i * K + k] * Vt[(size_t)k * dv + c];
            out[(size_t)i * dv + c] = num / den;
        }
    }
    rc = 0;
done:
    free(gq);
    free(gk);
    free(Vt);
    free(Z);
    return rc;
}

/*
 * One head of the backward pass: gradients of a loss L with respect to Qx, Kx,
 * V, mu, omega and alpha, given dO = dL/dO.  Section 4.1 fixes its structure
 * (the extraction of the paper lacks Appendix D): the upstream gradient g at a
 * responsibility vector enters the scores through the softmax Jacobian,
 * Eq. (17)-(18), ds_{i,k} = gamma_{i,k} (g_{i,k} - sum_j gamma_{i,j} g_{i,j});
 * every quantity that enters a score then collects sum_i sum_k ds_{i,k}
 * ds_{i,k}/dtheta, Eq. (19), with the score of Eq. (16) differentiated by hand:
 *   d s_{i,k} / d mu_k      =  Sigma_k^{-1} (x_i - mu_k)                 Eq. (20)
 *   d s_{i,k} / d x_i       = -Sigma_k^{-1} (x_i - mu_k)                 section 4.3
 *   d s_{i,k} / d var_{k,m} = (1/2) ((x_im - mu_km)^2 / var_km^2 - 1 / var_km)
 *   d s_{i,k} / d log pi_k  = 1
 * then var through Eq. (14) (d softplus / d omega = sigmoid(omega)) and
 * log pi through Eq. (15) (the log-softmax Jacobian).  The memory operations
 * are differentiated as the products they are: with den_i = gamma^Q_i . Z + eps
 * and O_i = gamma^Q_i Vt / den_i (Eq. 7-8), a_i = dO_i / den_i and
 * b_i = -(dO_i . O_i) / den_i give
 *   g^Q_i = Vt a_i + Z b_i,
 *   R = sum_i gamma^Q_i a_i^T,  r = sum_i gamma^Q_i b_i   (over the rows that read the memory),
 *   g^K_j = R v_j + r,  dV_j = R^T gamma^K_j.
 * causal = 1 uses the prefix memory of Eq. (6b)/(8b): row i reads the memory of
 * rows j <= i, so key j collects R and r over the rows i >= j (a suffix sum).
 * Every output is overwritten.  Layouts as for the forward: dQx, dKx [N, d],
 * dV [N, dv], dmu, domega [K, d], dalpha [K].
 */
int gma_oracle_backward_head(int N, int d, int K, int dv, const double *Qx, const double *Kx,
                             const double *V, const double *mu, const double *omega,
                             const double *alpha, double var_floor, double eps, int causal,
                             const double *dO, double *dQx, double *dKx, double *dV, double *dmu,
                             double *domega, double *dalpha)
{
    if (N < 0 || d <= 0 || K <= 0 || dv <= 0) return 1;
    size_t nk = (size_t)N * K, kdv = (size_t)K * dv, kd = (size_t)K * d;
    double *gq = (double *)malloc(sizeof(double) * (nk ? nk : 1));
    double *gk = (double *)malloc(sizeof(double) * (nk ? nk : 1));
    double *dgq = (double *)calloc(nk ? nk : 1, sizeof(double));
    double *dgk = (double *)calloc(nk ? nk : 1, sizeof(double));
    double *a = (double *)calloc((size_t)(N ? N : 1) * dv, sizeof(double));
    double *b = (double *)calloc(N ? N : 1, sizeof(double));
    double *Vt = (double *)calloc(kdv, sizeof(double));
    double *Z = (double *)calloc(K, sizeof(double));
    double *R = (double *)calloc(kdv, sizeof(double));
    double *r = (double *)calloc(K, sizeof(double));
    double *var = (double *)malloc(sizeof(double) * kd);
    double *dvar = (double *)calloc(kd, sizeof(double));
    double *dlogpi = (double *)calloc(K, sizeof(double));
    double *logpi = (double *)malloc(sizeof(double) * K);
    int rc = 2;
    if (!gq || !gk || !dgq || !dgk || !a || !b || !Vt || !Z || !R || !r || !var || !dvar || !dlogpi || !logpi)
        goto done;
    rc = gma_oracle_responsibilities(N, d, K, Qx, mu, omega, alpha, var_floor, gq);
    if (rc) goto done;
    rc = gma_oracle_responsibilities(N, d, K, Kx, mu, omega, alpha, var_floor, gk);
    if (rc) goto done;
    for (size_t e = 0; e < kd; ++e) var[e] = variance_from_omega(omega[e], var_floor);
    log_priors(K, alpha, logpi);

    /* Eq. (5)-(6) over the whole sequence (bidirectional); the causal memory grows below. */
    if (!causal)
        for (int j = 0; j < N; ++j)
            for (int k = 0; k < K; ++k) {
                double g = gk[(size_t)j * K + k];
                Z[k] += g;
                for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g * V[(size_t)j * dv + c];
            }
    /* the read of each row (Eq. 7-8 or 8b) and its gradient with respect to gamma^Q_i */
    for (int i = 0; i < N; ++i) {
        if (causal)
            for (int k = 0; k < K; ++k) {
                double g = gk[(size_t)i * K + k];
                Z[k] += g;
                for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g * V[(size_t)i * dv + c];
            }
        const double *gi = gq + (size_t)i * K;
        double den = eps;
        for (int k = 0; k < K; ++k) den += gi[k] * Z[k];
        double dot = 0.0;
        for (int c = 0; c < dv; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gi[k] * Vt[(size_t)k * dv + c];
            dot += dO[(size_t)i * dv + c] * (num / den);
            a[(size_t)i * dv + c] = dO[(size_t)i * dv + c] / den;
        }
        b[i] = -dot / den;
        for (int k = 0; k < K; ++k) {
            double g = Z[k] * b[i];
            for (int c = 0; c < dv; ++c) g += Vt[(size_t)k * dv + c] * a[(size_t)i * dv + c];
            dgq[(size_t)i * K + k] = g;
        }
    }
    /* R, r over the rows that read key j's memory; g^K_j and dV_j */
    if (!causal)
        for (int i = 0; i < N; ++i)
            for (int k = 0; k < K; ++k) {
                double g = gq[(size_t)i * K + k];
                r[k] += g * b[i];
                for (int c = 0; c < dv; ++c) R[(size_t)k * dv + c] += g * a[(size_t)i * dv + c];
            }
    for (int j = N - 1; j >= 0; --j) {
        if (causal)
            for (int k = 0; k < K; ++k) {
                double g = gq[(size_t)j * K + k];
                r[k] += g * b[j];
                for (int c = 0; c < dv; ++c) R[(size_t)k * dv + c] += g * a[(size_t)j * dv + c];
            }
        for (int k = 0; k < K; ++k) {
            double g = r[k];
            for (int c = 0; c < dv; ++c) g += R[(size_t)k * dv + c] * V[(size_t)j * dv + c];
            dgk[(size_t)j * K + k] = g;
        }
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int k = 0; k < K; ++k) s += R[(size_t)k * dv + c] * gk[(size_t)j * K + k];
            dV[(size_t)j * dv + c] = s;
        }
    }
    /* Eq. (18) then Eq. (19)-(20) for the query rows and the key rows alike */
    for (size_t e = 0; e < kd; ++e) dmu[e] = 0.0;
    for (int side = 0; side < 2; ++side) {
        const double *X = side ? Kx : Qx;
        const double *gam = side ? gk : gq;
        const double *dg = side ? dgk : dgq;
        double *dX = side ? dKx : dQx;
        for (int i = 0; i < N; ++i) {
            const double *gi = gam + (size_t)i * K, *dgi = dg + (size_t)i * K;
            double mean = 0.0;
            for (int k = 0; k < K; ++k) mean += gi[k] * dgi[k];
            for (int m = 0; m < d; ++m) dX[(size_t)i * d + m] = 0.0;
            for (int k = 0; k < K; ++k) {
                double ds = gi[k] * (dgi[k] - mean);
                dlogpi[k] += ds;
                for (int m = 0; m < d; ++m) {
                    double diff = X[(size_t)i * d + m] - mu[(size_t)k * d + m];
                    double vk = var[(size_t)k * d + m];
                    dX[(size_t)i * d + m] -= ds * diff / vk;
                    dmu[(size_t)k * d + m] += ds * diff / vk;
                    dvar[(size_t)k * d + m] += ds * 0.5 * (diff * diff / (vk * vk) - 1.0 / vk);
                }
            }
        }
    }
    /* Eq. (14): d var / d omega = sigmoid(omega); Eq. (15): the log-softmax Jacobian */
    for (size_t e = 0; e < kd; ++e) domega[e] = dvar[e] / (1.0 + exp(-omega[e]));
    {
        double tot = 0.0;
        for (int k = 0; k < K; ++k) tot += dlogpi[k];
        for (int k = 0; k < K; ++k) dalpha[k] = dlogpi[k] - exp(logpi[k]) * tot;
    }
    rc = 0;
done:
    free(gq); free(gk); free(dgq); free(dgk); free(a); free(b); free(Vt); free(Z); free(R); free(r);
    free(var); free(dvar); free(dlogpi); free(logpi);
    return rc;
}

/*
 * Input projections (section 3.1, Eq. 4): for every batch entry b and head h,
 *   Qx[b, h] = X[b] Wq[h],   Kx[b, h] = X[b] Wk[h],   V[b, h] = X[b] Wv[h],
 * with X [B, N, D], Wq and Wk [H, D, d], Wv [H, D, dv], and the results in the
 * [B, H, N, .] layout of the forward's inputs.  Each entry is a D-term dot product
 * summed in order of the model dimension.
 */
int gma_oracle_project(int B, int N, int D, int H, int d, int dv, const double *X, const double *Wq,
                       const double *Wk, const double *Wv, double *Qx, double *Kx, double *V)
{
    if (B < 0 || N < 0 || D <= 0 || H <= 0 || d <= 0 || dv <= 0) return 1;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < N; ++i) {
                const double *x = X + ((size_t)b * N + i) * D;
                const size_t row = ((size_t)b * H + h) * N + i;
                for (int c = 0; c < d; ++c) {
                    double q = 0.0, k = 0.0;
                    for (int m = 0; m < D; ++m) {
                        q += x[m] * Wq[((size_t)h * D + m) * d + c];
                        k += x[m] * Wk[((size_t)h * D + m) * d + c];
                    }
                    Qx[row * d + c] = q;
                    Kx[row * d + c] = k;
                }
                for (int c = 0; c < dv; ++c) {
                    double v = 0.0;
                    for (int m = 0; m < D; ++m) v += x[m] * Wv[((size_t)h * D + m) * dv + c];
                    V[row * dv + c] = v;
                }
            }
    return 0;
}
