/*
 * kdn_oracle.c -- plain fp64 CPU oracle for the Kalman Delta Network mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Source: "Kalman Delta Networks: Uncertainty-aware Associative Memory"
 * (Bui, Huang, Ying, arXiv:2609.07816v1), as summarised by its reading notes
 * and by its paperlayer summary.  The recurrence is run token by token, in the
 * order the paper states it, with no chunking, blocking or reordering:
 *
 *   Diagonal KDN (Sec. 4.1, Eq. 23-27; information scaling Eq. 60-65):
 *     a      = exp(log_alpha_t)                       (D_t = diag(a))
 *     p_hat  = a^2 * p + omega_t                      predictive variances
 *     S_hat  = diag(a) S                              predicted memory
 *     z      = sum_i p_hat_i k_i^2
 *     kappa  = p_hat * k / (r_t + z)                  Kalman gain
 *     delta  = v_t - S_hat^T k_t                      innovation
 *     S      = S_hat + kappa delta^T                  exact one-step mean
 *     o_t    = S^T q_t                                read AFTER the write
 *     u      = (mu / r_t) k * k
 *     p      = p_hat / (1 + u * p_hat)                scaled reverse-KL update
 *
 *   Isotropic KDN (Sec. 4.2, Eq. 40; App. C):
 *     a_bar  = (1/d_k) sum_i a_i^2                    trace projection
 *     b_hat  = a_bar * b + omega_t
 *     beta   = b_hat / (r_t + b_hat ||k||^2),  kappa = beta k
 *     (mean path identical to the diagonal case, D_t = diag(a))
 *     u      = mu ||k||^2 / (d_k r_t),  b = b_hat / (1 + u b_hat)
 *
 * The mean path is the exact Kalman mean for the retained (diagonal or
 * isotropic) predictive prior (Sec. 3.2, Eq. 12-17).  The gain uses the
 * predictive variance p_hat, before the mu-scaled update, so mu changes only
 * later gains (App. B).
 *
 * Layouts (row-major, innermost last):
 *   q, k, log_alpha            [B,T,H,dk]
 *   v, o                       [B,T,H,dv]
 *   omega                      [B,T,H,dk] (diagonal) or [B,T,H] (isotropic)
 *   r                          [B,T,H]    observation-noise VARIANCE
 *   S0, S_T                    [B,H,dk,dv]  (row = key channel)
 *   p0, p_T                    [B,H,dk] (diagonal) or [B,H] (isotropic)
 *   kappa_out (optional)       [B,T,H,dk]
 *   phat_out  (optional)       [B,T,H,dk] (diagonal) or [B,T,H] (isotropic)
 * S0 == NULL means S_0 = 0; p0 == NULL means p_0 = 1.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_DIAG = 0, ORACLE_ISO = 1 };

typedef struct {
    int variant, B, T, H, dk, dv;
    double mu;
    const double *q, *k, *v, *log_alpha, *omega, *r, *S0, *p0;
    double *o, *S_T, *p_T, *kappa_out, *phat_out;
    int next;             /* next (b,h) pair to run, guarded by lock */
    pthread_mutex_t lock;
    int failed;
} oracle_job;

/* One (b,h) sequence, token by token. Returns 0 on success. */
static int run_sequence(oracle_job *J, int b, int h)
{
    const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    const int nu = (J->variant == ORACLE_DIAG) ? dk : 1;   /* uncertainty entries */
    double *S = malloc(sizeof(double) * (size_t)dk * dv);
    double *p = malloc(sizeof(double) * (size_t)nu);
    double *a = malloc(sizeof(double) * (size_t)dk);
    double *phat = malloc(sizeof(double) * (size_t)nu);
    double *kappa = malloc(sizeof(double) * (size_t)dk);
    double *delta = malloc(sizeof(double) * (size_t)dv);
    if (!S || !p || !a || !phat || !kappa || !delta) {
        free(S); free(p); free(a); free(phat); free(kappa); free(delta);
        return 1;
    }
    const size_t sidx = ((size_t)b * H + h) * (size_t)dk * dv;
    const size_t pidx = ((size_t)b * H + h) * (size_t)nu;
    for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = J->S0 ? J->S0[sidx + e] : 0.0;
    for (int i = 0; i < nu; ++i) p[i] = J->p0 ? J->p0[pidx + i] : 1.0;

    for (int t = 0; t < T; ++t) {
        const size_t th = ((size_t)b * T + t) * H + h;     /* token-head index */
        const double *qt = J->q + th * dk, *kt = J->k + th * dk;
        const double *vt = J->v + th * dv, *lat = J->log_alpha + th * dk;
        const double rt = J->r[th];
        double *ot = J->o + th * dv;

        /* predict: D_t = diag(a), covariance decays by a^2 */
        for (int i = 0; i < dk; ++i) a[i] = exp(lat[i]);
        double knorm2 = 0.0;
        for (int i = 0; i < dk; ++i) knorm2 += kt[i] * kt[i];
        if (J->variant == ORACLE_DIAG) {
            const double *omt = J->omega + th * dk;
            for (int i = 0; i < dk; ++i) phat[i] = a[i] * a[i] * p[i] + omt[i];
        } else {
            double abar = 0.0;
            for (int i = 0; i < dk; ++i) abar += a[i] * a[i];
            abar /= (double)dk;
            phat[0] = abar * p[0] + J->omega[th];
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a[i];

        /* gain */
        if (J->variant == ORACLE_DIAG) {
            double z = 0.0;
            for (int i = 0; i < dk; ++i) z += phat[i] * kt[i] * kt[i];
            for (int i = 0; i < dk; ++i) kappa[i] = phat[i] * kt[i] / (rt + z);
        } else {
            const double beta = phat[0] / (rt + phat[0] * knorm2);
            for (int i = 0; i < dk; ++i) kappa[i] = beta * kt[i];
        }

        /* innovation against the predicted memory, then the write */
        for (int j = 0; j < dv; ++j) {
            double pred = 0.0;
            for (int i = 0; i < dk; ++i) pred += S[(size_t)i * dv + j] * kt[i];
            delta[j] = vt[j] - pred;
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kappa[i] * delta[j];

        /* readout from the post-write memory */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];
            ot[j] = acc;
        }

        if (J->kappa_out)
            for (int i = 0; i < dk; ++i) J->kappa_out[th * dk + i] = kappa[i];
        if (J->phat_out)
            for (int i = 0; i < nu; ++i) J->phat_out[th * nu + i] = phat[i];

        /* information-scaled posterior variance, used only by later tokens */
        if (J->variant == ORACLE_DIAG) {
            for (int i = 0; i < dk; ++i) {
                const double u = (J->mu / rt) * kt[i] * kt[i];
                p[i] = phat[i] / (1.0 + u * phat[i]);
            }
        } else {
            const double u = J->mu * knorm2 / ((double)dk * rt);
            p[0] = phat[0] / (1.0 + u * phat[0]);
        }
    }

    for (size_t e = 0; e < (size_t)dk * dv; ++e) J->S_T[sidx + e] = S[e];
    for (int i = 0; i < nu; ++i) J->p_T[pidx + i] = p[i];
    free(S); free(p); free(a); free(phat); free(kappa); free(delta);
    return 0;
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int w = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (w >= J->B * J->H) break;
        if (run_sequence(J, w / J->H, w % J->H)) {
            pthread_mutex_lock(&J->lock);
            J->failed = 1;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

/* Number of host threads the oracle uses when asked for "all cores". */
int kdn_oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Run the full recurrence over every (b,h) sequence.  Sequences are
 * independent (each head has its own memory and uncertainty), so they are
 * spread over `nthreads` host threads (<= 0 means all online cores).
 * Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 */
int kdn_oracle_forward(int variant, int B, int T, int H, int dk, int dv, double mu,
                       const double *q, const double *k, const double *v,
                       const double *log_alpha, const double *omega, const double *r,
                       const double *S0, const double *p0,
                       double *o, double *S_T, double *p_T,
                       double *kappa_out, double *phat_out, int nthreads)
{
    if ((variant != ORACLE_DIAG && variant != ORACLE_ISO) || B < 0 || T < 0 || H < 0 ||
        dk <= 0 || dv <= 0)
        return 1;
    if (!q || !k || !v || !log_alpha || !omega || !r || !o || !S_T || !p_T) return 1;
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.variant = variant; J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.mu = mu;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.omega = omega; J.r = r;
    J.S0 = S0; J.p0 = p0; J.o = o; J.S_T = S_T; J.p_T = p_T;
    J.kappa_out = kappa_out; J.phat_out = phat_out;
    pthread_mutex_init(&J.lock, NULL);
    int n = nthreads > 0 ? nthreads : kdn_oracle_default_threads();
    if (n > B * H) n = B * H;
    if (n < 1) n = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)n);
    if (!th) { pthread_mutex_destroy(&J.lock); return 2; }
    int started = 0;
    for (int i = 0; i < n; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? 2 : 0;
}
