/*
 * pkda_oracle.c -- plain fp64 CPU oracle for the preconditioned delta rule
 * with per-channel decay (PKDA), and its no-decay relatives PDN and PGDN.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests and the CPU baseline leg of the benchmark
 * use it.  It shares no code, header, table or constant with the CUDA
 * library.
 *
 * Source: "Preconditioned DeltaNet" reading notes (arXiv:2604.21100v1):
 * Sec. 2.2 (apply-to-key, Theorem 3.1 / Eq. 3-5), Sec. 2.3 (diagonal key
 * statistic, App. C.2), Sec. 2.4 (the trained parameterisation, Eq. 9) and
 * Sec. 2.5 (forgetting: PDN D = I, PGDN D = alpha I, PKDA D = Diag(alpha)).
 * The pages write the memory as S (d_v x d_k) with right-multiplied decay;
 * here S is stored transposed (d_k x d_v, row = key channel), so the decay
 * multiplies from the left.  Per (b,h), token by token:
 *
 *   a      = exp(log_alpha_t)               D_t = diag(a)
 *   write key k_til (selected by `mode`):
 *     SQUASH     (Eq. 9):  A = alpha_p_t A + beta_p_t (k * k)   (this token included)
 *                          rho = log(max(A, floor)) - mu_h
 *                          s   = rho / (1 + |rho|)              (softsign)
 *                          k_til = exp(-log(x) s) * k           (scale in [1/x, x])
 *     DIAG_ATK   (Sec. 2.3, App. C.2): the diagonal statistic A (A_0 = lambda)
 *                          taken BEFORE this token: k_til = (k / A) / (1 + sum k^2 / A),
 *                          then A = A + k * k
 *     EXACT_ATK  (Sec. 2.2, Thm 3.1): dense P (P_0 = I / lambda):
 *                          k_til = P k / (1 + k^T P k),
 *                          then P = P - P k k^T P / (1 + k^T P k)  (Sherman-Morrison)
 *   S_hat  = diag(a) S
 *   delta  = v_t - S_hat^T k_t              the residual uses the READ key k
 *   S      = S_hat + beta_t k_til delta^T   the write uses the WRITE key k_til
 *   o_t    = S^T q_t                        read after the write
 *
 * Only SQUASH is the trained model; the two ATK modes are the pages' exact
 * theory and serve to pin the shared write/readout path (with beta = 1 and no
 * decay, EXACT_ATK must reproduce ridge regression exactly, Thm 3.1).
 *
 * The statistic floor: the pages leave the guard on log(0) open; this oracle
 * takes log(max(A, 1e-20)).
 *
 * Layouts (row-major, innermost last):
 *   q, k, log_alpha          [B,T,H,dk]
 *   v, o                     [B,T,H,dv]
 *   beta, alpha_p, beta_p    [B,T,H]
 *   center (mu_h)            [H]
 *   S0, S_T                  [B,H,dk,dv]
 *   A0, A_T                  [B,H,dk]   (SQUASH, DIAG_ATK); unused by EXACT_ATK
 *   kappa_out (optional)     [B,T,H,dk] = beta_t * k_til_t
 * S0 == NULL means S_0 = 0; A0 == NULL means A_0 = 0 (SQUASH) or lambda (DIAG_ATK).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { PKDA_SQUASH = 0, PKDA_DIAG_ATK = 1, PKDA_EXACT_ATK = 2 };

static const double kStatFloor = 1e-20;

typedef struct {
    int mode, B, T, H, dk, dv;
    double x, lam;
    const double *q, *k, *v, *log_alpha, *beta, *alpha_p, *beta_p, *center, *S0, *A0;
    double *o, *S_T, *A_T, *kappa_out;
    int next;
    pthread_mutex_t lock;
    int failed;
} pkda_job;

static int run_sequence(pkda_job *J, int b, int h)
{
    const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    double *S = malloc(sizeof(double) * (size_t)dk * dv);
    double *A = malloc(sizeof(double) * (size_t)dk);
    double *kt = malloc(sizeof(double) * (size_t)dk);
    double *delta = malloc(sizeof(double) * (size_t)dv);
    double *P = NULL, *Pk = NULL;
    if (J->mode == PKDA_EXACT_ATK) {
        P = malloc(sizeof(double) * (size_t)dk * dk);
        Pk = malloc(sizeof(double) * (size_t)dk);
    }
    if (!S || !A || !kt || !delta || (J->mode == PKDA_EXACT_ATK && (!P || !Pk))) {
        free(S); free(A); free(kt); free(delta); free(P); free(Pk);
        return 1;
    }
    const size_t sidx = ((size_t)b * H + h) * (size_t)dk * dv;
    const size_t aidx = ((size_t)b * H + h) * (size_t)dk;
    for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = J->S0 ? J->S0[sidx + e] : 0.0;
    for (int i = 0; i < dk; ++i)
        A[i] = J->A0 ? J->A0[aidx + i] : (J->mode == PKDA_DIAG_ATK ? J->lam : 0.0);
    if (P)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dk; ++j) P[(size_t)i * dk + j] = (i == j) ? 1.0 / J->lam : 0.0;
    const double mu = J->center ? J->center[h] : 0.0;
    const double logx = log(J->x);

    for (int t = 0; t < T; ++t) {
        const size_t th = ((size_t)b * T + t) * H + h;
        const double *qt = J->q + th * dk, *kv = J->k + th * dk;
        const double *vt = J->v + th * dv, *lat = J->log_alpha + th * dk;
        const double bt = J->beta[th];
        double *ot = J->o + th * dv;

        /* write key */
        if (J->mode == PKDA_SQUASH) {
            const double ap = J->alpha_p[th], bp = J->beta_p[th];
            for (int i = 0; i < dk; ++i) {
                A[i] = ap * A[i] + bp * kv[i] * kv[i];
                const double rho = log(A[i] > kStatFloor ? A[i] : kStatFloor) - mu;
                const double s = rho / (1.0 + fabs(rho));
                kt[i] = exp(-logx * s) * kv[i];
            }
        } else if (J->mode == PKDA_DIAG_ATK) {
            double kpk = 0.0;
            for (int i = 0; i < dk; ++i) kpk += kv[i] * kv[i] / A[i];
            for (int i = 0; i < dk; ++i) kt[i] = (kv[i] / A[i]) / (1.0 + kpk);
            for (int i = 0; i < dk; ++i) A[i] += kv[i] * kv[i];
        } else {
            double kpk = 0.0;
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += P[(size_t)i * dk + j] * kv[j];
                Pk[i] = acc;
                kpk += kv[i] * acc;
            }
            for (int i = 0; i < dk; ++i) kt[i] = Pk[i] / (1.0 + kpk);
            /* P is symmetric: P k k^T P = Pk Pk^T */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dk; ++j) P[(size_t)i * dk + j] -= Pk[i] * Pk[j] / (1.0 + kpk);
        }

        /* decay, residual with the read key, write with the write key */
        for (int i = 0; i < dk; ++i) {
            const double a = exp(lat[i]);
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
        }
        for (int j = 0; j < dv; ++j) {
            double pred = 0.0;
            for (int i = 0; i < dk; ++i) pred += S[(size_t)i * dv + j] * kv[i];
            delta[j] = vt[j] - pred;
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += bt * kt[i] * delta[j];

        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];
            ot[j] = acc;
        }
        if (J->kappa_out)
            for (int i = 0; i < dk; ++i) J->kappa_out[th * dk + i] = bt * kt[i];
    }

    for (size_t e = 0; e < (size_t)dk * dv; ++e) J->S_T[sidx + e] = S[e];
    if (J->A_T)
        for (int i = 0; i < dk; ++i) J->A_T[aidx + i] = A[i];
    free(S); free(A); free(kt); free(delta); free(P); free(Pk);
    return 0;
}

static void *worker(void *arg)
{
    pkda_job *J = (pkda_job *)arg;
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

/*
 * Run the recurrence over every (b,h) sequence on `nthreads` host threads
 * (<= 0: all online cores).  alpha_p, beta_p and center are read by SQUASH
 * only.  Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 */
int pkda_oracle_forward(int mode, int B, int T, int H, int dk, int dv, double x, double lam,
                        const double *q, const double *k, const double *v,
                        const double *log_alpha, const double *beta, const double *alpha_p,
                        const double *beta_p, const double *center,
                        const double *S0, const double *A0,
                        double *o, double *S_T, double *A_T, double *kappa_out, int nthreads)
{
    if (mode < PKDA_SQUASH || mode > PKDA_EXACT_ATK || B < 0 || T < 0 || H < 0 || dk <= 0 ||
        dv <= 0 || !(x > 0.0) || !(lam > 0.0))
        return 1;
    if (!q || !k || !v || !log_alpha || !beta || !o || !S_T) return 1;
    if (mode == PKDA_SQUASH && (!alpha_p || !beta_p || !center)) return 1;
    pkda_job J;
    memset(&J, 0, sizeof(J));
    J.mode = mode; J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.x = x; J.lam = lam;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta; J.alpha_p = alpha_p;
    J.beta_p = beta_p; J.center = center; J.S0 = S0; J.A0 = A0;
    J.o = o; J.S_T = S_T; J.A_T = A_T; J.kappa_out = kappa_out;
    pthread_mutex_init(&J.lock, NULL);
    long nc = sysconf(_SC_NPROCESSORS_ONLN);
    int n = nthreads > 0 ? nthreads : (nc > 0 ? (int)nc : 1);
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
