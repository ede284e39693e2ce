/*
 * kda_oracle.c -- plain, sequential fp64 CPU oracle for the KDA recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  The CUDA path
 * never calls, links or includes anything from here, and this file includes
 * nothing from the CUDA path.
 *
 * What it computes (sources are the pages' titles and sections):
 *
 *  - "Noyaux KDA et FlashKDA", section "Le conflit fondamental": each head
 *    keeps a fixed-size state S in R^{dk x dv}.  The update equation itself is
 *    not printed on any page; the form implemented is the gated delta rule
 *        S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T,
 *        o_t = scale * S_t^T q_t,
 *    with Diag(exp g) acting on the key (dk) axis, g per channel.
 *  - same page, section "Le role de la decroissance bornee": the per-channel
 *    log-decay is floored at g_min = -5, applied per token and per channel.
 *  - same page, section "Le parallelisme de contexte intra-appareil", and
 *    "Dentro de los esfuerzos de optimizacion de Kimi K3", section 5
 *    ("KDA: paralelizar el prellenado..."): a segment's state transition is an
 *    affine map S -> M S + N that does not depend on the incoming state, and
 *    transitions compose exactly.
 *  - "Noyaux d'inference", section 1 ("Le decodage KDA"), subsections "La
 *    solution : rejouer plutot que sauvegarder" and "La fusion": the verify
 *    step replays accepted draft tokens from their cached projected inputs,
 *    then runs short conv -> input norm -> gating -> recurrence -> output norm
 *    over the replayed tokens, the bonus token and the next draft window, and
 *    writes back the state reached after the bonus token.
 *  - "Dentro de los esfuerzos...", "Nota tecnica: Precision del KDA y memoria
 *    on-chip": the intra-chunk dependency matrix is inverted by substituting
 *    earlier corrections into later ones (unit lower-triangular inverse).
 *
 * Everything is fp64, one loop nest per (sequence, head) or (request, head).
 * OpenMP only spreads those independent units over host threads; within a
 * unit the arithmetic runs token by token in the pages' order.
 *
 * Readings where the pages are silent (all listed in the design notes):
 * softplus/sigmoid gates, L2 input norm with eps, per-head RMSNorm output
 * norm with a [dv] weight, depthwise causal conv whose last tap multiplies
 * the current token, tail = the W-1 most recent pre-conv rows (oldest first),
 * optional SiLU after the conv.
 *
 * Parity pins for each function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

/* ------------------------------------------------------------------------- */
/* One token of the gated delta rule on one head's state S[dk][dv].           */
/*   S' = Diag(exp(max(g, g_min))) S                                          */
/*   erase = 1:  S = S' - b k (k^T S') + b k v^T   ((I - b k k^T) S' + b k v^T)*/
/*   erase = 0:  S = S' + b k v^T   (no-erase switch, used only by the pins   */
/*               that reduce the rule to decayed / plain linear attention)    */
/* tmp must hold dv doubles.                                                 */
/* ------------------------------------------------------------------------- */
/* The floor max(g, g_min).  A NaN log-decay takes the floor (the pages say  */
/* nothing of NaN; IEEE maximum returns the non-NaN operand).                */
static double floor_g(double g, double g_min) { return g >= g_min ? g : g_min; }

static void kda_token(int dk, int dv, double *S, const double *k, const double *v,
                      const double *g, double beta, double g_min, int erase,
                      double *tmp)
{
    for (int i = 0; i < dk; ++i) {
        double gi = floor_g(g[i], g_min);
        double d = exp(gi);
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= d;
    }
    if (erase) {
        /* tmp = S'^T k */
        for (int j = 0; j < dv; ++j) tmp[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) tmp[j] += k[i] * S[(size_t)i * dv + j];
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] += beta * k[i] * (v[j] - tmp[j]);
    } else {
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += beta * k[i] * v[j];
    }
}

/* o = scale * S^T q */
static void kda_readout(int dk, int dv, const double *S, const double *q, double scale,
                        double *o)
{
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) o[j] += q[i] * S[(size_t)i * dv + j];
    for (int j = 0; j < dv; ++j) o[j] *= scale;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* Prefill: N sequences packed along T by cu_seqlens[N+1].                    */
/* q,k [T][H][dk], v [T][H][dv], g [T][H][dk], beta [T][H]                    */
/* S0 [N][H][dk][dv] or NULL (zero), o [T][H][dv], S_final [N][H][dk][dv] or  */
/* NULL.  head_mask[H] (or NULL = all): heads with mask 0 are skipped and     */
/* their outputs left untouched (lets tests sample heads at full size).       */
/* ------------------------------------------------------------------------- */
int oracle_kda_prefill(int N, int T, int H, int dk, int dv, const int32_t *cu_seqlens,
                       const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const double *S0, double *o, double *S_final,
                       double scale, double g_min, int erase, const uint8_t *head_mask,
                       int nthreads)
{
    if (N < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return ORACLE_EINVAL;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return ORACLE_EINVAL;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return ORACLE_EINVAL;
    set_threads(nthreads);
    long units = (long)N * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        int n = (int)(u / H), h = (int)(u % H);
        if (head_mask && !head_mask[h]) continue;
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *tmp = (double *)malloc(sizeof(double) * (size_t)dv);
        size_t so = ((size_t)n * H + h) * (size_t)dk * dv;
        if (S0) memcpy(S, S0 + so, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            size_t th = (size_t)t * H + h;
            kda_token(dk, dv, S, k + th * dk, v + th * dv, g + th * dk, beta[th], g_min,
                      erase, tmp);
            kda_readout(dk, dv, S, q + th * dk, scale, o + th * dv);
        }
        if (S_final) memcpy(S_final + so, S, sizeof(double) * (size_t)dk * dv);
        free(S);
        free(tmp);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Backward of the prefill (reverse mode of the token recurrence above; the   */
/* pages name the backward pass as the other use of the chunk kernel,         */
/* "Noyaux KDA et FlashKDA", section "FlashKDA : le noyau par blocs"), per    */
/* (sequence, head).  Inputs as oracle_kda_prefill (erase on) plus            */
/* do_ [T][H][dv] and dS_final [N][H][dk][dv] (or NULL: zero).  Outputs       */
/* dq, dk_ [T][H][dk], dv_ [T][H][dv], dg [T][H][dk] (gradient w.r.t. the raw */
/* g: zero where the floor holds, g < g_min), dbeta [T][H], dS0 [N][H][dk][dv] */
/* (or NULL).  Per token (S before, S' after, D = Diag(e^{max(g, g_min)}),    */
/* X = D S, p = X^T k, u = beta (v - p), S' = X + k u^T, o = scale S'^T q),   */
/* with G the gradient w.r.t. S' coming from later tokens:                   */
/*   G += scale q do^T;  dq = scale S' do;  du = G^T k;  dv = beta du;        */
/*   dbeta = du . (v - p);  dk = G u - beta X du;  dX = G - beta k du^T;      */
/*   dg_i = sum_j dX_ij X_ij  (where g_i >= g_min);  G <- D dX.               */
/* Every forward state of a sequence is kept (small cases only).             */
/* ------------------------------------------------------------------------- */
int oracle_kda_backward(int N, int T, int H, int dk, int dv, const int32_t *cu_seqlens,
                        const double *q, const double *k, const double *v, const double *g,
                        const double *beta, const double *S0, const double *do_,
                        const double *dS_final, double *dq, double *dk_, double *dv_, double *dg,
                        double *dbeta, double *dS0, double scale, double g_min, int nthreads)
{
    if (N < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return ORACLE_EINVAL;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return ORACLE_EINVAL;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return ORACLE_EINVAL;
    set_threads(nthreads);
    const size_t DD = (size_t)dk * dv;
    long units = (long)N * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long un = 0; un < units; ++un) {
        int n = (int)(un / H), h = (int)(un % H);
        int t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - t0;
        size_t so = ((size_t)n * H + h) * DD;
        double *Sall = (double *)malloc(sizeof(double) * DD * (size_t)(L + 1));
        double *G = (double *)malloc(sizeof(double) * DD);
        double *X = (double *)malloc(sizeof(double) * DD);
        double *tmp = (double *)malloc(sizeof(double) * (size_t)dv * 4);
        double *p = tmp, *u = tmp + dv, *du = tmp + 2 * dv;
        if (S0) memcpy(Sall, S0 + so, sizeof(double) * DD);
        else memset(Sall, 0, sizeof(double) * DD);
        for (int t = 0; t < L; ++t) {
            size_t th = (size_t)(t0 + t) * H + h;
            memcpy(Sall + DD * (t + 1), Sall + DD * t, sizeof(double) * DD);
            kda_token(dk, dv, Sall + DD * (t + 1), k + th * dk, v + th * dv, g + th * dk, beta[th], g_min, 1,
                      tmp + 3 * dv);
        }
        if (dS_final) memcpy(G, dS_final + so, sizeof(double) * DD);
        else memset(G, 0, sizeof(double) * DD);
        for (int t = L - 1; t >= 0; --t) {
            size_t th = (size_t)(t0 + t) * H + h;
            const double *qt = q + th * dk, *kt = k + th * dk, *vt = v + th * dv, *gt = g + th * dk;
            const double *dot = do_ + th * dv, *Sp = Sall + DD * t, *Sn = Sall + DD * (t + 1);
            double bt = beta[th];
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] += scale * qt[i] * dot[j];
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += Sn[(size_t)i * dv + j] * dot[j];
                dq[th * dk + i] = scale * acc;
            }
            for (int i = 0; i < dk; ++i) {
                double gi = floor_g(gt[i], g_min);
                double d = exp(gi);
                for (int j = 0; j < dv; ++j) X[(size_t)i * dv + j] = d * Sp[(size_t)i * dv + j];
            }
            for (int j = 0; j < dv; ++j) {
                double pj = 0.0, dj = 0.0;
                for (int i = 0; i < dk; ++i) {
                    pj += X[(size_t)i * dv + j] * kt[i];
                    dj += G[(size_t)i * dv + j] * kt[i];
                }
                p[j] = pj;
                u[j] = bt * (vt[j] - pj);
                du[j] = dj;
            }
            double db = 0.0;
            for (int j = 0; j < dv; ++j) {
                dv_[th * dv + j] = bt * du[j];
                db += du[j] * (vt[j] - p[j]);
            }
            dbeta[th] = db;
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j)
                    acc += G[(size_t)i * dv + j] * u[j] - bt * X[(size_t)i * dv + j] * du[j];
                dk_[th * dk + i] = acc;
            }
            for (int i = 0; i < dk; ++i) {
                double gi = floor_g(gt[i], g_min);
                double d = exp(gi), acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    double dx = G[(size_t)i * dv + j] - bt * kt[i] * du[j];
                    acc += dx * X[(size_t)i * dv + j];
                    G[(size_t)i * dv + j] = d * dx;
                }
                dg[th * dk + i] = (gt[i] < g_min) ? 0.0 : acc;
            }
        }
        if (dS0) memcpy(dS0 + so, G, sizeof(double) * DD);
        free(Sall);
        free(G);
        free(X);
        free(tmp);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Segment transition over tokens [0, T) of the given arrays, per head:       */
/*   M = A_T ... A_1,  A_t = (I - b_t k_t k_t^T) Diag(exp g_t)   [H][dk][dk]  */
/*   N = state reached from S = 0                                 [H][dk][dv] */
/* M is built by applying each A_t on the left, starting from the identity:   */
/* that is the token step with v = 0 on a dk x dk "state".                    */
/* ------------------------------------------------------------------------- */
int oracle_segment_transition(int T, int H, int dk, int dv, const double *k, const double *v,
                              const double *g, const double *beta, double g_min, double *M,
                              double *Nmat, int nthreads)
{
    if (T < 0 || H <= 0 || dk <= 0 || dv <= 0) return ORACLE_EINVAL;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        double *Mh = M + (size_t)h * dk * dk;
        double *Nh = Nmat + (size_t)h * dk * dv;
        double *zero_v = (double *)calloc((size_t)dk, sizeof(double));
        double *tmp = (double *)malloc(sizeof(double) * (size_t)(dk > dv ? dk : dv));
        memset(Mh, 0, sizeof(double) * (size_t)dk * dk);
        for (int i = 0; i < dk; ++i) Mh[(size_t)i * dk + i] = 1.0;
        memset(Nh, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < T; ++t) {
            size_t th = (size_t)t * H + h;
            kda_token(dk, dk, Mh, k + th * dk, zero_v, g + th * dk, beta[th], g_min, 1, tmp);
            kda_token(dk, dv, Nh, k + th * dk, v + th * dv, g + th * dk, beta[th], g_min, 1, tmp);
        }
        free(zero_v);
        free(tmp);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Ordered composition, per head:  S_in[p] = S_{p-1},  S_p = M_p S_{p-1} + N_p */
/* with S_{-1} = S0 (or 0).  M [P][H][dk][dk], Nmat/S_in [P][H][dk][dv],       */
/* S0/S_final [H][dk][dv] (either may be NULL).                               */
/* ------------------------------------------------------------------------- */
int oracle_segment_compose(int P, int H, int dk, int dv, const double *M, const double *Nmat,
                           const double *S0, double *S_in, double *S_final)
{
    if (P < 0 || H <= 0 || dk <= 0 || dv <= 0) return ORACLE_EINVAL;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    for (int h = 0; h < H; ++h) {
        if (S0) memcpy(S, S0 + (size_t)h * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int p = 0; p < P; ++p) {
            const double *Mp = M + ((size_t)p * H + h) * dk * dk;
            const double *Np = Nmat + ((size_t)p * H + h) * dk * dv;
            if (S_in) memcpy(S_in + ((size_t)p * H + h) * dk * dv, S, sizeof(double) * (size_t)dk * dv);
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) {
                    double acc = Np[(size_t)i * dv + j];
                    for (int r = 0; r < dk; ++r) acc += Mp[(size_t)i * dk + r] * S[(size_t)r * dv + j];
                    Sn[(size_t)i * dv + j] = acc;
                }
            memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
        }
        if (S_final) memcpy(S_final + (size_t)h * dk * dv, S, sizeof(double) * (size_t)dk * dv);
    }
    free(S);
    free(Sn);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* T = (I + A)^{-1} for a strictly lower-triangular n x n A (row-major), by   */
/* forward substitution: each row of T takes its direct coefficient and the   */
/* corrections that reach it through every earlier position.                 */
/* ------------------------------------------------------------------------- */
int oracle_unit_lower_inverse(int n, const double *A, double *Tm)
{
    if (n < 0) return ORACLE_EINVAL;
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < n; ++j) {
            double x = (i == j) ? 1.0 : 0.0;
            if (j < i)
                for (int m = j; m < i; ++m) x -= A[(size_t)i * n + m] * Tm[(size_t)m * n + j];
            Tm[(size_t)i * n + j] = x;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Chunk-form (WY) reference of one head over one sequence, fp64, chunk C.    */
/* Used only to pin the chunk algebra against the token-by-token definition;  */
/* the decays are exponentiated directly (fp64 has the range for it).         */
/* Within a chunk, with gamma_t = sum_{r<=t} max(g_r, g_min) per channel:     */
/*   A[t,s] = b_t sum_c k_tc k_sc exp(gamma_tc - gamma_sc)      (s <  t)      */
/*   B[t,s] =     sum_c q_tc k_sc exp(gamma_tc - gamma_sc)      (s <= t)      */
/*   Tm = (I + A)^{-1};  W = Tm diag(b) (K . e^gamma);  Ut = Tm diag(b) V      */
/*   U = Ut - W S;  O = scale((Q . e^gamma) S + B U)                           */
/*   S <- Diag(e^gamma_last) S + (K . e^{gamma_last - gamma})^T U             */
/* q,k [T][dk], v [T][dv], g [T][dk], beta [T]; S in/out [dk][dv]; o [T][dv]. */
/* ------------------------------------------------------------------------- */
int oracle_chunk_form_head(int T, int dk, int dv, int C, const double *q, const double *k,
                           const double *v, const double *g, const double *beta, double *S,
                           double *o, double scale, double g_min)
{
    if (T < 0 || dk <= 0 || dv <= 0 || C <= 0) return ORACLE_EINVAL;
    double *gam = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *B = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *Tm = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    for (int c0 = 0; c0 < T; c0 += C) {
        int L = (T - c0 < C) ? (T - c0) : C;
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int t = 0; t < L; ++t) {
                double gi = g[(size_t)(c0 + t) * dk + i];
                acc += floor_g(gi, g_min);
                gam[(size_t)t * dk + i] = acc;
            }
        }
        for (int t = 0; t < L; ++t)
            for (int s = 0; s < L; ++s) {
                double a = 0.0, b = 0.0;
                if (s <= t)
                    for (int c = 0; c < dk; ++c) {
                        double e = exp(gam[(size_t)t * dk + c] - gam[(size_t)s * dk + c]);
                        a += k[(size_t)(c0 + t) * dk + c] * k[(size_t)(c0 + s) * dk + c] * e;
                        b += q[(size_t)(c0 + t) * dk + c] * k[(size_t)(c0 + s) * dk + c] * e;
                    }
                A[(size_t)t * L + s] = (s < t) ? beta[c0 + t] * a : 0.0;
                B[(size_t)t * L + s] = (s <= t) ? b : 0.0;
            }
        oracle_unit_lower_inverse(L, A, Tm);
        for (int t = 0; t < L; ++t) {
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int s = 0; s <= t; ++s)
                    acc += Tm[(size_t)t * L + s] * beta[c0 + s] * k[(size_t)(c0 + s) * dk + c] *
                           exp(gam[(size_t)s * dk + c]);
                W[(size_t)t * dk + c] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int s = 0; s <= t; ++s)
                    acc += Tm[(size_t)t * L + s] * beta[c0 + s] * v[(size_t)(c0 + s) * dv + j];
                for (int c = 0; c < dk; ++c) acc -= W[(size_t)t * dk + c] * S[(size_t)c * dv + j];
                U[(size_t)t * dv + j] = acc;
            }
        }
        for (int t = 0; t < L; ++t)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c)
                    acc += q[(size_t)(c0 + t) * dk + c] * exp(gam[(size_t)t * dk + c]) *
                           S[(size_t)c * dv + j];
                for (int s = 0; s <= t; ++s) acc += B[(size_t)t * L + s] * U[(size_t)s * dv + j];
                o[(size_t)(c0 + t) * dv + j] = scale * acc;
            }
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j) {
                double acc = exp(gam[(size_t)(L - 1) * dk + c]) * S[(size_t)c * dv + j];
                for (int s = 0; s < L; ++s)
                    acc += k[(size_t)(c0 + s) * dk + c] *
                           exp(gam[(size_t)(L - 1) * dk + c] - gam[(size_t)s * dk + c]) *
                           U[(size_t)s * dv + j];
                Sn[(size_t)c * dv + j] = acc;
            }
        memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
    }
    free(gam); free(A); free(B); free(Tm); free(W); free(U); free(Sn);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Speculative-decode verify with replay ("Noyaux d'inference", section 1).   */
/*                                                                            */
/* Channel layout of a pre-conv projected row (Cq = H*(2*dk+dv) channels):    */
/*   [ q: H*dk | k: H*dk | v: H*dv ], head h owns q[h*dk..], k[h*dk..],       */
/*   v[h*dv..] inside each part.                                             */
/* state [R][H][dk][dv]      in/out (write-back = state after the bonus token) */
/* tail  [R][W-1][Cq]        in/out (the W-1 most recent pre-conv rows,        */
/*                           oldest first; written back after the bonus)       */
/* conv_w [Cq][W]            y_t = sum_j w[c][j] x_{t-(W-1)+j}                 */
/* cached_qkv [R][Wd][Cq], cached_g [R][Wd][H*dk], cached_b [R][Wd][H]         */
/* new_qkv [R][Wd+1][Cq], new_g [R][Wd+1][H*dk], new_b [R][Wd+1][H]            */
/*                           (row 0 = bonus token, rows 1..Wd = next drafts)   */
/* accepted [R] in [0, Wd];  out_w [dv];  o [R][Wd+1][H][dv]                  */
/* draft_len [R] in [0, Wd] or NULL (every request has Wd drafts): request r  */
/* has new rows 0..draft_len[r] (ragged batches, "Dentro de los esfuerzos de  */
/* optimizacion de Kimi K3", section 5: irregular batches keep a dynamic      */
/* path); its o rows past draft_len[r] are not written.                       */
/* Token order per request: cached rows 0..a-1 (replayed), new row 0 (bonus), */
/* new rows 1..Wd (drafts).  Per token: conv (+SiLU if conv_act) -> L2 norm   */
/* of q and k over dk -> g = max(-softplus(g_raw), g_min), b = sigmoid(b_raw) */
/* -> recurrence step -> for bonus and drafts o = RMSNorm(scale S^T q) * w.   */
/* Requests with an out-of-range accepted or draft length are skipped         */
/* entirely (state, tail and o untouched) and counted in the return value.    */
/* ------------------------------------------------------------------------- */
static double softplus(double x) { return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x))); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

struct verify_args {
    int R, H, dk, dv, W, Wd, conv_act;
    double eps_in, eps_out, scale, g_min;
    const double *conv_w, *cached_qkv, *cached_g, *cached_b, *new_qkv, *new_g, *new_b, *out_w;
    const int32_t *accepted;
};

/* Pointer to the pre-conv row at sequence position p of request r, where the
 * sequence is tail rows (positions 0..W-2), then cached rows 0..a-1, then new
 * rows 0..Wd.  Returns NULL past the end. */
static const double *seq_row(const struct verify_args *A, const double *tail_r, int r, int a,
                             int p)
{
    int Cq = A->H * (2 * A->dk + A->dv);
    int nt = A->W - 1;
    if (p < nt) return tail_r + (size_t)p * Cq;
    p -= nt;
    if (p < a) return A->cached_qkv + ((size_t)r * A->Wd + p) * Cq;
    p -= a;
    if (p <= A->Wd) return A->new_qkv + ((size_t)r * (A->Wd + 1) + p) * Cq;
    return NULL;
}

/* Process request r, head h for the first n_tok tokens of its verify
 * sequence.  Writes o rows for tokens at positions >= a (bonus/drafts), the
 * state after token index a into state_out, and nothing else. */
static void verify_unit(const struct verify_args *A, int r, int h, int a, int n_tok,
                        const double *S_in, const double *tail_r, double *S_wb, double *o)
{
    int dk = A->dk, dv = A->dv, W = A->W, H = A->H;
    int Cq = H * (2 * dk + dv);
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)dv);
    double *qv = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kv = (double *)malloc(sizeof(double) * (size_t)dk);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *gv = (double *)malloc(sizeof(double) * (size_t)dk);
    double *ov = (double *)malloc(sizeof(double) * (size_t)dv);
    memcpy(S, S_in, sizeof(double) * (size_t)dk * dv);
    int cq0 = h * dk, ck0 = H * dk + h * dk, cv0 = 2 * H * dk + h * dv;
    for (int t = 0; t < n_tok; ++t) {
        int p = (W - 1) + t; /* sequence position of this token */
        /* short conv over the W most recent pre-conv rows, per channel */
        for (int c = 0; c < dk + dk + dv; ++c) {
            int ch = c < dk ? cq0 + c : (c < 2 * dk ? ck0 + (c - dk) : cv0 + (c - 2 * dk));
            double y = 0.0;
            for (int j = 0; j < W; ++j) {
                const double *row = seq_row(A, tail_r, r, a, p - (W - 1) + j);
                y += A->conv_w[(size_t)ch * W + j] * row[ch];
            }
            if (A->conv_act) y = y * sigmoid(y);
            if (c < dk) qv[c] = y;
            else if (c < 2 * dk) kv[c - dk] = y;
            else vv[c - 2 * dk] = y;
        }
        (void)Cq;
        /* input norm: L2 over dk for q and k */
        double sq = 0.0, sk = 0.0;
        for (int i = 0; i < dk; ++i) { sq += qv[i] * qv[i]; sk += kv[i] * kv[i]; }
        double rq = 1.0 / sqrt(sq + A->eps_in), rk = 1.0 / sqrt(sk + A->eps_in);
        for (int i = 0; i < dk; ++i) { qv[i] *= rq; kv[i] *= rk; }
        /* gating */
        const double *graw, *braw;
        if (t < a) {
            graw = A->cached_g + ((size_t)r * A->Wd + t) * (size_t)(H * dk) + (size_t)h * dk;
            braw = A->cached_b + ((size_t)r * A->Wd + t) * H + h;
        } else {
            graw = A->new_g + ((size_t)r * (A->Wd + 1) + (t - a)) * (size_t)(H * dk) + (size_t)h * dk;
            braw = A->new_b + ((size_t)r * (A->Wd + 1) + (t - a)) * H + h;
        }
        for (int i = 0; i < dk; ++i) {
            double gg = -softplus(graw[i]);
            gv[i] = floor_g(gg, A->g_min);
        }
        double beta = sigmoid(*braw);
        kda_token(dk, dv, S, kv, vv, gv, beta, A->g_min, 1, tmp);
        if (t >= a && o) {
            kda_readout(dk, dv, S, qv, A->scale, ov);
            double ms = 0.0;
            for (int j = 0; j < dv; ++j) ms += ov[j] * ov[j];
            double rr = 1.0 / sqrt(ms / dv + A->eps_out);
            double *dst = o + (((size_t)r * (A->Wd + 1) + (t - a)) * H + h) * dv;
            for (int j = 0; j < dv; ++j) dst[j] = ov[j] * rr * A->out_w[j];
        }
        if (t == a && S_wb) memcpy(S_wb, S, sizeof(double) * (size_t)dk * dv);
    }
    free(S); free(tmp); free(qv); free(kv); free(vv); free(gv); free(ov);
}

static int request_ok(const int32_t *accepted, const int32_t *draft_len, int Wd, int r)
{
    if (accepted[r] < 0 || accepted[r] > Wd) return 0;
    if (draft_len && (draft_len[r] < 0 || draft_len[r] > Wd)) return 0;
    return 1;
}

int oracle_decode_verify_ragged(int R, int H, int dk, int dv, int W, int Wd, double *state,
                                double *tail, const double *conv_w, const double *cached_qkv,
                                const double *cached_g, const double *cached_b,
                                const int32_t *accepted, const int32_t *draft_len,
                                const double *new_qkv, const double *new_g, const double *new_b,
                                const double *out_w, double eps_in, double eps_out, int conv_act,
                                double *o, double scale, double g_min, int nthreads)
{
    if (R < 0 || H <= 0 || dk <= 0 || dv <= 0 || W < 1 || Wd < 0) return ORACLE_EINVAL;
    struct verify_args A = {R, H, dk, dv, W, Wd, conv_act, eps_in, eps_out, scale, g_min,
                            conv_w, cached_qkv, cached_g, cached_b, new_qkv, new_g, new_b,
                            out_w, accepted};
    int Cq = H * (2 * dk + dv);
    int bad = 0;
    for (int r = 0; r < R; ++r)
        if (!request_ok(accepted, draft_len, Wd, r)) ++bad;
    set_threads(nthreads);
    /* heads read the shared old tail, so the new tails are written after all
       heads of a request are done: copy old tails first */
    double *old_tail = (double *)malloc(sizeof(double) * (size_t)R * (W - 1) * Cq + 1);
    memcpy(old_tail, tail, sizeof(double) * (size_t)R * (W - 1) * Cq);
    long units = (long)R * H;
#pragma omp parallel for schedule(dynamic, 4)
    for (long u = 0; u < units; ++u) {
        int r = (int)(u / H), h = (int)(u % H);
        if (!request_ok(accepted, draft_len, Wd, r)) continue;
        int a = accepted[r], d = draft_len ? draft_len[r] : Wd;
        double *S = state + ((size_t)r * H + h) * (size_t)dk * dv;
        verify_unit(&A, r, h, a, a + 1 + d, S, old_tail + (size_t)r * (W - 1) * Cq, S, o);
    }
    /* conv tail write-back: the W-1 most recent pre-conv rows up to and
       including the bonus token, oldest first (a bitwise copy) */
    for (int r = 0; r < R; ++r) {
        if (!request_ok(accepted, draft_len, Wd, r)) continue;
        int a = accepted[r];
        const double *tr = old_tail + (size_t)r * (W - 1) * Cq;
        int last = (W - 1) + a; /* sequence position of the bonus token */
        for (int m = 0; m < W - 1; ++m) {
            const double *row = seq_row(&A, tr, r, a, last - (W - 2) + m);
            memcpy(tail + ((size_t)r * (W - 1) + m) * Cq, row, sizeof(double) * (size_t)Cq);
        }
    }
    free(old_tail);
    return bad;
}

int oracle_decode_verify(int R, int H, int dk, int dv, int W, int Wd, double *state,
                         double *tail, const double *conv_w, const double *cached_qkv,
                         const double *cached_g, const double *cached_b,
                         const int32_t *accepted, const double *new_qkv, const double *new_g,
                         const double *new_b, const double *out_w, double eps_in,
                         double eps_out, int conv_act, double *o, double scale, double g_min,
                         int nthreads)
{
    return oracle_decode_verify_ragged(R, H, dk, dv, W, Wd, state, tail, conv_w, cached_qkv,
                                       cached_g, cached_b, accepted, NULL, new_qkv, new_g, new_b,
                                       out_w, eps_in, eps_out, conv_act, o, scale, g_min, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Non-speculative decoding of the same tokens, one token per call: for each  */
/* request, feed the a accepted cached rows and then the bonus row one at a   */
/* time through a single-token decode step that reads and writes the state    */
/* and the conv tail after every token (as a plain decoder would).  Arrays as */
/* in oracle_decode_verify; o receives the bonus row only ([R][H][dv]).       */
/* ------------------------------------------------------------------------- */
static void decode_one(int H, int dk, int dv, int W, double *state_r, double *tail_r,
                       const double *conv_w, const double *x, const double *graw,
                       const double *braw, const double *out_w, double eps_in, double eps_out,
                       int conv_act, double *o_r, double scale, double g_min)
{
    int Cq = H * (2 * dk + dv);
    /* the sequence for a single token is tail ++ [x]: reuse the verify path
       with a = 0, no drafts, a one-row "new" block */
    struct verify_args A = {1, H, dk, dv, W, 0, conv_act, eps_in, eps_out, scale, g_min,
                            conv_w, NULL, NULL, NULL, x, graw, braw, out_w, NULL};
    for (int h = 0; h < H; ++h) {
        double *S = state_r + (size_t)h * dk * dv;
        verify_unit(&A, 0, h, 0, 1, S, tail_r, S, o_r);
    }
    /* shift the tail by one row */
    if (W > 1) {
        memmove(tail_r, tail_r + Cq, sizeof(double) * (size_t)(W - 2) * Cq);
        memcpy(tail_r + (size_t)(W - 2) * Cq, x, sizeof(double) * (size_t)Cq);
    }
}

int oracle_decode_stepwise(int R, int H, int dk, int dv, int W, int Wd, double *state,
                           double *tail, const double *conv_w, const double *cached_qkv,
                           const double *cached_g, const double *cached_b,
                           const int32_t *accepted, const double *new_qkv, const double *new_g,
                           const double *new_b, const double *out_w, double eps_in,
                           double eps_out, int conv_act, double *o_bonus, double scale,
                           double g_min)
{
    if (R < 0 || H <= 0 || dk <= 0 || dv <= 0 || W < 1 || Wd < 0) return ORACLE_EINVAL;
    int Cq = H * (2 * dk + dv);
    int bad = 0;
    for (int r = 0; r < R; ++r) {
        int a = accepted[r];
        if (a < 0 || a > Wd) { ++bad; continue; }
        double *st = state + (size_t)r * H * dk * dv;
        double *tl = tail + (size_t)r * (W - 1) * Cq;
        double *orow = o_bonus + (size_t)r * H * dv;
        for (int t = 0; t <= a; ++t) {
            const double *x, *gr, *br;
            if (t < a) {
                x = cached_qkv + ((size_t)r * Wd + t) * Cq;
                gr = cached_g + ((size_t)r * Wd + t) * (size_t)(H * dk);
                br = cached_b + ((size_t)r * Wd + t) * H;
            } else {
                x = new_qkv + ((size_t)r * (Wd + 1)) * Cq;
                gr = new_g + ((size_t)r * (Wd + 1)) * (size_t)(H * dk);
                br = new_b + ((size_t)r * (Wd + 1)) * H;
            }
            decode_one(H, dk, dv, W, st, tl, conv_w, x, gr, br, out_w, eps_in, eps_out,
                       conv_act, orow, scale, g_min);
        }
    }
    return bad;
}
