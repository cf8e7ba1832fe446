/*
 * efla_oracle.c -- plain fp64 CPU oracle for Exact Flow Linear Attention (EFLA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes (source: "Exact Flow Linear Attention: Exact Solution from
 * Continuous-Time Dynamics", gist.science summary of arXiv 2512.12602, page es,
 * section "Metodologia", items 1-3; the ja/de/fr pages repeat the same items):
 *
 *   ODE (item 1):          dS/dt = -A_t S + b_t,  A_t = k_t k_t^T,  b_t = k_t v_t^T
 *   closed form (item 2):  exp(-beta_t A_t) = I - ((1 - exp(-beta_t lambda_t))/lambda_t) A_t,
 *                          lambda_t = ||k_t||^2
 *   update rule (item 3):  S_t = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T,
 *                          alpha_t = (1 - exp(-beta_t lambda_t)) / lambda_t
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - read-out o_t = S_t^T q_t with the state *after* token t's update;
 *   - state S is d_k x d_v (the shape of k v^T), row index = key dimension;
 *   - alpha -> beta as lambda -> 0 (the limit of the formula; exactly beta at lambda = 0);
 *   - "Euler" mode (alpha := beta) is the delta rule that the pages name as the
 *     explicit Euler step of the same ODE (page es, "Contribuciones Clave", first item).
 *
 * The recurrence is evaluated token by token, in order, with no chunking,
 * blocking or reordering.  The backward pass is reverse-mode differentiation
 * of that same loop (derived by calculus; the pages give no backward pass),
 * recomputing states from checkpoints every EFLA_ORACLE_SEG tokens.
 *
 * Layouts (all row-major, contiguous, double):
 *   q, k [B,H,L,dk]   v, o [B,H,L,dv]   beta [B,H,L]   S [B,H,dk,dv]
 *
 * Parallelism: OpenMP over the B*H independent sequences when compiled with
 * -fopenmp; nthreads <= 0 means "all available".
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define EFLA_ORACLE_SEG 64

/* ---------------------------------------------------------------- alpha -- */

/* alpha(beta, lambda) = (1 - e^{-beta lambda}) / lambda, written as
 * beta * phi(x) with x = beta*lambda and phi(x) = (1 - e^{-x})/x, phi(0) = 1.
 * expm1 keeps the small-x end accurate.  euler != 0 gives alpha = beta. */
double efla_oracle_alpha(double beta, double lambda, int euler)
{
    if (euler) return beta;
    double x = beta * lambda;
    if (x == 0.0) return beta;
    return beta * (-expm1(-x) / x);
}

/* d alpha / d beta = e^{-beta lambda}  (1 in Euler mode). */
double efla_oracle_dalpha_dbeta(double beta, double lambda, int euler)
{
    if (euler) return 1.0;
    return exp(-beta * lambda);
}

/* d alpha / d lambda = beta^2 phi'(x),  phi'(x) = (x e^{-x} + expm1(-x)) / x^2.
 * For |x| < 0.05 the Taylor series of phi' is summed instead:
 *   phi'(x) = sum_{n>=1} n (-x)^{n-1} (-1) / (n+1)!   (i.e. -1/2 + x/3 - x^2/8 + ...). */
double efla_oracle_dalpha_dlambda(double beta, double lambda, int euler)
{
    if (euler) return 0.0;
    double x = beta * lambda;
    double dphi;
    if (fabs(x) < 0.05) {
        double fact = 2.0;      /* (n+1)! for n = 1 */
        double xp = 1.0;        /* x^{n-1} */
        double sgn = -1.0;      /* (-1)^n */
        dphi = 0.0;
        for (int n = 1; n <= 14; ++n) {
            dphi += sgn * (double)n * xp / fact;
            xp *= x;
            sgn = -sgn;
            fact *= (double)(n + 2);
        }
    } else {
        dphi = (x * exp(-x) + expm1(-x)) / (x * x);
    }
    return beta * beta * dphi;
}

/* ------------------------------------------------------------ one token -- */

/* S <- S + alpha k r^T with r = v - S^T k  (identical to the update rule);
 * r_out receives r.  Returns alpha. */
static double token_update(int dk, int dv, const double* k, const double* v,
                           double beta, double* S, double* r_out, int euler)
{
    double lambda = 0.0;
    for (int i = 0; i < dk; ++i) lambda += k[i] * k[i];
    double a = efla_oracle_alpha(beta, lambda, euler);
    for (int j = 0; j < dv; ++j) r_out[j] = v[j];
    for (int i = 0; i < dk; ++i) {
        const double* row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) r_out[j] -= row[j] * k[i];
    }
    for (int i = 0; i < dk; ++i) {
        double c = a * k[i];
        double* row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) row[j] += c * r_out[j];
    }
    return a;
}

/* o = S^T q */
static void readout(int dk, int dv, const double* S, const double* q, double* o)
{
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        const double* row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) o[j] += row[j] * q[i];
    }
}

static int pick_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int efla_oracle_max_threads(void)
{
    return pick_threads(0);
}

/* ---------------------------------------------------------------- forward -- */

/* S0 may be NULL (zeros).  S_final may be NULL.  o may be NULL. */
int efla_oracle_fwd(int B, int H, int L, int dk, int dv,
                    const double* q, const double* k, const double* v,
                    const double* beta, const double* S0,
                    double* o, double* S_final, int euler, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0) return 1;
    long nh = (long)B * H;
    size_t ss = (size_t)dk * dv;
    int nt = pick_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : err)
    for (long h = 0; h < nh; ++h) {
        double* S = (double*)malloc(ss * sizeof(double));
        double* r = (double*)malloc((size_t)dv * sizeof(double));
        if (!S || !r) { free(S); free(r); err |= 1; continue; }
        if (S0) memcpy(S, S0 + h * ss, ss * sizeof(double));
        else memset(S, 0, ss * sizeof(double));
        for (int t = 0; t < L; ++t) {
            size_t tok = (size_t)h * L + t;
            token_update(dk, dv, k + tok * dk, v + tok * dv, beta[tok], S, r, euler);
            if (o) readout(dk, dv, S, q + tok * dk, o + tok * dv);
        }
        if (S_final) memcpy(S_final + h * ss, S, ss * sizeof(double));
        free(S);
        free(r);
    }
    return err;
}

/* One decode step per sequence: S [B,H,dk,dv] updated in place, o [B,H,dv].
 * q, k [B,H,dk], v [B,H,dv], beta [B,H].  Same arithmetic as forward with L = 1. */
int efla_oracle_step(int B, int H, int dk, int dv,
                     const double* q, const double* k, const double* v,
                     const double* beta, double* S, double* o, int euler, int nthreads)
{
    return efla_oracle_fwd(B, H, 1, dk, dv, q, k, v, beta, S, o, S, euler, nthreads);
}

/* --------------------------------------------------------------- backward -- */

/* Reverse-mode gradient of   sum(o * dO) + sum(S_final * dS_final)
 * with respect to q, k, v, beta and S0.  dS_final and S0 may be NULL (zeros);
 * dS0 may be NULL.  Per token, with G = dLoss/dS_t flowing backwards:
 *   o_t = S_t^T q_t            ->  dq_t = S_t dO_t,       G += q_t dO_t^T
 *   r = v_t - S_{t-1}^T k_t,  S_t = S_{t-1} + alpha k r^T
 *                              ->  dalpha = k^T G r,      dr = alpha G^T k
 *                                  dk_t  = alpha G r - S_{t-1} dr + 2 dalpha (dalpha/dlambda) k_t
 *                                  dv_t  = dr,            dbeta_t = dalpha (dalpha/dbeta)
 *                                  G    <- G - k dr^T     (gradient reaching S_{t-1})
 */
int efla_oracle_bwd(int B, int H, int L, int dk, int dv,
                    const double* q, const double* k, const double* v,
                    const double* beta, const double* S0,
                    const double* dO, const double* dS_final,
                    double* dq, double* dk_out, double* dv_out, double* dbeta,
                    double* dS0, int euler, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0) return 1;
    long nh = (long)B * H;
    size_t ss = (size_t)dk * dv;
    int nseg = (L + EFLA_ORACLE_SEG - 1) / EFLA_ORACLE_SEG;
    int nt = pick_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : err)
    for (long h = 0; h < nh; ++h) {
        double* ck = (double*)malloc((size_t)(nseg > 0 ? nseg : 1) * ss * sizeof(double));
        double* buf = (double*)malloc((size_t)(EFLA_ORACLE_SEG + 1) * ss * sizeof(double));
        double* G = (double*)malloc(ss * sizeof(double));
        double* r = (double*)malloc((size_t)dv * sizeof(double));
        double* dr = (double*)malloc((size_t)dv * sizeof(double));
        double* Gr = (double*)malloc((size_t)dk * sizeof(double));
        if (!ck || !buf || !G || !r || !dr || !Gr) {
            free(ck); free(buf); free(G); free(r); free(dr); free(Gr);
            err |= 1;
            continue;
        }
        /* forward pass, keeping the state before every segment */
        double* S = buf;
        if (S0) memcpy(S, S0 + h * ss, ss * sizeof(double));
        else memset(S, 0, ss * sizeof(double));
        for (int t = 0; t < L; ++t) {
            if (t % EFLA_ORACLE_SEG == 0)
                memcpy(ck + (size_t)(t / EFLA_ORACLE_SEG) * ss, S, ss * sizeof(double));
            size_t tok = (size_t)h * L + t;
            token_update(dk, dv, k + tok * dk, v + tok * dv, beta[tok], S, r, euler);
        }
        if (dS_final) memcpy(G, dS_final + h * ss, ss * sizeof(double));
        else memset(G, 0, ss * sizeof(double));

        for (int s = nseg - 1; s >= 0; --s) {
            int t0 = s * EFLA_ORACLE_SEG;
            int t1 = t0 + EFLA_ORACLE_SEG;
            if (t1 > L) t1 = L;
            /* buf[m] = state before token t0+m, m = 0..t1-t0 */
            memcpy(buf, ck + (size_t)s * ss, ss * sizeof(double));
            for (int t = t0; t < t1; ++t) {
                double* nxt = buf + (size_t)(t - t0 + 1) * ss;
                memcpy(nxt, buf + (size_t)(t - t0) * ss, ss * sizeof(double));
                size_t tok = (size_t)h * L + t;
                token_update(dk, dv, k + tok * dk, v + tok * dv, beta[tok], nxt, r, euler);
            }
            for (int t = t1 - 1; t >= t0; --t) {
                size_t tok = (size_t)h * L + t;
                const double* St = buf + (size_t)(t - t0 + 1) * ss;
                const double* Sp = buf + (size_t)(t - t0) * ss;
                const double* qt = q + tok * dk;
                const double* kt = k + tok * dk;
                const double* vt = v + tok * dv;
                const double* gt = dO + tok * dv;
                /* read-out */
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) acc += St[(size_t)i * dv + j] * gt[j];
                    dq[tok * dk + i] = acc;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] += qt[i] * gt[j];
                /* update */
                double lambda = 0.0;
                for (int i = 0; i < dk; ++i) lambda += kt[i] * kt[i];
                double bt = beta[tok];
                double a = efla_oracle_alpha(bt, lambda, euler);
                for (int j = 0; j < dv; ++j) r[j] = vt[j];
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) r[j] -= Sp[(size_t)i * dv + j] * kt[i];
                double da = 0.0;
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) acc += G[(size_t)i * dv + j] * r[j];
                    Gr[i] = acc;
                    da += kt[i] * acc;
                }
                for (int j = 0; j < dv; ++j) dr[j] = 0.0;
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) dr[j] += G[(size_t)i * dv + j] * kt[i];
                for (int j = 0; j < dv; ++j) dr[j] *= a;
                double dl = da * efla_oracle_dalpha_dlambda(bt, lambda, euler);
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) acc += Sp[(size_t)i * dv + j] * dr[j];
                    dk_out[tok * dk + i] = a * Gr[i] - acc + 2.0 * dl * kt[i];
                }
                for (int j = 0; j < dv; ++j) dv_out[tok * dv + j] = dr[j];
                dbeta[tok] = da * efla_oracle_dalpha_dbeta(bt, lambda, euler);
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] -= kt[i] * dr[j];
            }
        }
        if (dS0) memcpy(dS0 + h * ss, G, ss * sizeof(double));
        free(ck); free(buf); free(G); free(r); free(dr); free(Gr);
    }
    return err;
}
