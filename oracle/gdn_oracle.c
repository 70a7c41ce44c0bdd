/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle of the chunkwise gated-delta
 * prefill core (dense and event-sparse forms).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it is used by the tests, by the smoke check and by the
 * benchmark's CPU-baseline leg.  It shares no code with the CUDA library.
 *
 * Source of every formula: "SparseGDN: Chunk Sparse in Linear Attention",
 * Chinese reading notes (cc.laoqi.cc), which paraphrase the paper section by
 * section.  Section / equation numbers below are the paper's, as those notes
 * quote them.
 *
 * Notation (one value head h, its query/key head p = h/2, chunk c of L = 64
 * tokens, local token index i):
 *   g_{c,i}   within-chunk inclusive cumulative log2 retention   (Sec. 2.1)
 *   gamma_c   g at the chunk's last token                         (Sec. 2.1)
 *   A_Delta[t,s] = beta_t <k_t,k_s> 2^(g_t-g_s) [s<t],  M = I + A_Delta  (Sec. 2.3, Eqs. 5-6)
 *   U = M^-1 diag(beta) V,  W = M^-1 diag(beta 2^g) K                     (Eqs. 6, 8, 15)
 *   selected chunk:   U' = U - W S,  S+ = 2^gamma S + K^T (U' * 2^(gamma-g))  (Eqs. 1-2)
 *   unselected chunk: U' = U,        S+ = 2^gamma S                           (Eqs. 17-18)
 *   group (c, c+1) = (2r, 2r+1), entry state S_c:                             (Eqs. 22-24)
 *     O_c   = [2^g_c * (Q_c S_c) + A_cc U'_c] / sqrt(d)
 *     O_c+1 = [2^(g_c+1 + gamma_c) * (Q_c+1 S_c) + A_c+1,c U'_c + A_c+1,c+1 U'_c+1] / sqrt(d)
 *     A_cc[i,j] = <q_i,k_j> 2^(g_i - g_j) [j<=i];  A_c+1,c[i,j] = <q_i,k_j> 2^(g_c+1,i + gamma_c - g_c,j)
 *   chunk form (Eqs. 3-4): O_c = [2^g_c * (Q_c S_c) + A_cc U'_c] / sqrt(d) for every c.
 *   block-adjacent solver (Eq. 7): C_ii = M_ii^-1, C_i,i-1 = -C_ii M_i,i-1 C_i-1,i-1,
 *     every other 16x16 block zero; exact ("Full64") solver: C = M^-1.
 *   tail score (Eq. 9): s_c = ||U[48:64, :]||_F (Tail-16; the window W of Tail-W, W in
 *   {8, 16, 32, 64}, is the ablation axis of Sec. 3 / Fig. 10: the last W rows).
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *   - g is inclusive of token i's own gate (only then does Eq. 4's diagonal
 *     term carry weight 2^0 and Eqs. 5-6 match the token recurrence);
 *   - beta and g are per value head; q, k are per query/key head p = h/2;
 *   - 1/sqrt(d) scales both output terms; no other query scaling;
 *   - a partial last chunk of n < 64 tokens uses gamma = g at its last token
 *     and the tail window of its last min(16, n) tokens; the 16-token blocks
 *     of the solver are cut at n;
 *   - the state entering a group is the directly propagated state (the
 *     prefix-gap recovery of Eq. 21 is not used here, so it can be tested).
 *
 * Single-token decode (the state S_C returned for later autoregressive
 * decoding, Sec. 2.6): Eqs. 1-4 for a chunk of one token with log2 retention
 * a (so g = gamma = a, A_Delta is empty, M = 1):
 *   U = beta v,  W = beta 2^a k,  U' = U - W S,  S+ = 2^a S + k U'^T,
 *   o = [2^a (q^T S) + <q,k> U'] / sqrt(d).
 *
 * Exported entry points: gdn_oracle_prefill(), gdn_oracle_events(),
 * gdn_oracle_select(), gdn_oracle_decode().
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define LCH 64   /* chunk length L */
#define BLK 16   /* solver block size */

enum { SOLVER_EXACT = 0, SOLVER_BLOCK_ADJ = 1 };

typedef struct {
    int B, T, Nq, Nv, d, dv, solver;
    const double *q, *k, *v, *beta, *g, *h0;
    const unsigned char *mask; /* [B, Nv/2, C]; NULL = every chunk selected */
    double *o, *s_final;       /* required outputs */
    /* optional diagnostics (NULL to skip) */
    double *o_chunk, *u, *u_prime, *w, *s_in, *score, *cinv;
    int nthreads;
    int tail;                  /* rows of the tail-score window (16 by default) */
} job_t;

/* ---- small dense helpers (row-major, explicit sizes) --------------------- */

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* X = M^-1 for the n x n unit lower-triangular M, by forward substitution,
 * one column of the identity at a time. */
static void inverse_unit_lower(const double *M, int n, double *X)
{
    memset(X, 0, sizeof(double) * LCH * LCH);
    for (int j = 0; j < n; ++j) {
        for (int i = 0; i < n; ++i) {
            if (i < j) { X[i * LCH + j] = 0.0; continue; }
            if (i == j) { X[i * LCH + j] = 1.0; continue; }
            double acc = 0.0;
            for (int s = j; s < i; ++s) acc += M[i * LCH + s] * X[s * LCH + j];
            X[i * LCH + j] = -acc;
        }
    }
}

/* Block-adjacent approximation of M^-1 (Sec. 2.3, Eq. 7). */
static void inverse_block_adjacent(const double *M, int n, double *X)
{
    memset(X, 0, sizeof(double) * LCH * LCH);
    int nb = (n + BLK - 1) / BLK;
    /* diagonal blocks: C_ii = M_ii^-1 (forward substitution inside the block) */
    for (int bi = 0; bi < nb; ++bi) {
        int r0 = bi * BLK, r1 = r0 + BLK < n ? r0 + BLK : n;
        for (int j = r0; j < r1; ++j) {
            for (int i = j; i < r1; ++i) {
                if (i == j) { X[i * LCH + j] = 1.0; continue; }
                double acc = 0.0;
                for (int s = j; s < i; ++s) acc += M[i * LCH + s] * X[s * LCH + j];
                X[i * LCH + j] = -acc;
            }
        }
    }
    /* sub-diagonal blocks: C_i,i-1 = -C_ii M_i,i-1 C_i-1,i-1 */
    for (int bi = 1; bi < nb; ++bi) {
        int r0 = bi * BLK, r1 = r0 + BLK < n ? r0 + BLK : n;
        int c0 = (bi - 1) * BLK, c1 = c0 + BLK;
        double T1[BLK * BLK]; /* T1 = M_i,i-1 C_i-1,i-1 */
        for (int i = r0; i < r1; ++i)
            for (int j = c0; j < c1; ++j) {
                double acc = 0.0;
                for (int m = c0; m < c1; ++m) acc += M[i * LCH + m] * X[m * LCH + j];
                T1[(i - r0) * BLK + (j - c0)] = acc;
            }
        for (int i = r0; i < r1; ++i)
            for (int j = c0; j < c1; ++j) {
                double acc = 0.0;
                for (int m = r0; m < r1; ++m) acc += X[i * LCH + m] * T1[(m - r0) * BLK + (j - c0)];
                X[i * LCH + j] = -acc;
            }
    }
}

/* ---- one (b, value head) unit ------------------------------------------- */

typedef struct {
    /* per-chunk local copies */
    double *Qc, *Kc, *Vc, *bet, *gg;
    /* intra results */
    double *M, *Cm, *U, *W, *Up;
    /* previous chunk of the current group (for the odd chunk's cross term) */
    double *Qp, *Kp, *Up_prev, *gp;
    double *S, *Sgrp, *Sent; /* running state, group entry state, chunk entry state */
    double *tmp;
} scratch_t;

static void load_chunk(const job_t *J, int b, int h, int c, int n,
                       double *Qc, double *Kc, double *Vc, double *bet, double *gg)
{
    int p = h / 2, d = J->d, dv = J->dv;
    for (int i = 0; i < n; ++i) {
        size_t t = (size_t)c * LCH + i;
        size_t qk = (((size_t)b * J->T + t) * J->Nq + p) * d;
        size_t vv = (((size_t)b * J->T + t) * J->Nv + h) * dv;
        size_t sc = ((size_t)b * J->T + t) * J->Nv + h;
        memcpy(Qc + (size_t)i * d, J->q + qk, sizeof(double) * d);
        memcpy(Kc + (size_t)i * d, J->k + qk, sizeof(double) * d);
        memcpy(Vc + (size_t)i * dv, J->v + vv, sizeof(double) * dv);
        bet[i] = J->beta[sc];
        gg[i] = J->g[sc];
    }
}

/* Intra-chunk step (Sec. 2.3): M, the solver's C, U = C diag(beta) V,
 * W = C diag(beta 2^g) K. */
static void intra(const job_t *J, int n, scratch_t *X)
{
    int d = J->d, dv = J->dv;
    for (int t = 0; t < LCH; ++t)
        for (int s = 0; s < LCH; ++s) X->M[t * LCH + s] = 0.0;
    for (int t = 0; t < n; ++t) {
        X->M[t * LCH + t] = 1.0;
        for (int s = 0; s < t; ++s)
            X->M[t * LCH + s] = X->bet[t] * dot(X->Kc + (size_t)t * d, X->Kc + (size_t)s * d, d)
                                * exp2(X->gg[t] - X->gg[s]);
    }
    if (J->solver == SOLVER_EXACT) inverse_unit_lower(X->M, n, X->Cm);
    else inverse_block_adjacent(X->M, n, X->Cm);
    for (int t = 0; t < n; ++t) {
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int s = 0; s <= t; ++s) acc += X->Cm[t * LCH + s] * X->bet[s] * X->Vc[(size_t)s * dv + j];
            X->U[(size_t)t * dv + j] = acc;
        }
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int s = 0; s <= t; ++s)
                acc += X->Cm[t * LCH + s] * X->bet[s] * exp2(X->gg[s]) * X->Kc[(size_t)s * d + j];
            X->W[(size_t)t * d + j] = acc;
        }
    }
}

/* State read/write of one chunk (Eqs. 1-2 when selected, 17-18 otherwise). */
static void propagate(const job_t *J, int n, int selected, scratch_t *X)
{
    int d = J->d, dv = J->dv;
    double gam = X->gg[n - 1];
    if (selected) {
        for (int t = 0; t < n; ++t)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int m = 0; m < d; ++m) acc += X->W[(size_t)t * d + m] * X->S[(size_t)m * dv + j];
                X->Up[(size_t)t * dv + j] = X->U[(size_t)t * dv + j] - acc;
            }
        for (int m = 0; m < d; ++m)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int t = 0; t < n; ++t)
                    acc += X->Kc[(size_t)t * d + m] * X->Up[(size_t)t * dv + j] * exp2(gam - X->gg[t]);
                X->S[(size_t)m * dv + j] = exp2(gam) * X->S[(size_t)m * dv + j] + acc;
            }
    } else {
        memcpy(X->Up, X->U, sizeof(double) * (size_t)n * dv);
        for (size_t e = 0; e < (size_t)d * dv; ++e) X->S[e] = exp2(gam) * X->S[e];
    }
}

/* O rows for the tokens of one chunk given an entry state Sx and an extra
 * exponent `shift` on the state read (gamma_c for the odd chunk of a group).
 * Adds the local term A_cc U'_c.  out has stride dv, rows n. */
static void output_local(const job_t *J, int n, const double *Qc, const double *Kc, const double *Up,
                         const double *gg, const double *Sx, double shift, double *out)
{
    int d = J->d, dv = J->dv;
    double scale = 1.0 / sqrt((double)d);
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int m = 0; m < d; ++m) acc += Qc[(size_t)i * d + m] * Sx[(size_t)m * dv + j];
            out[(size_t)i * dv + j] = exp2(gg[i] + shift) * acc;
        }
        for (int s = 0; s <= i; ++s) {
            double a = dot(Qc + (size_t)i * d, Kc + (size_t)s * d, d) * exp2(gg[i] - gg[s]);
            for (int j = 0; j < dv; ++j) out[(size_t)i * dv + j] += a * Up[(size_t)s * dv + j];
        }
        for (int j = 0; j < dv; ++j) out[(size_t)i * dv + j] *= scale;
    }
}

static void store_rows(const job_t *J, double *dst, int b, int h, int c, int n, const double *src, int width)
{
    if (!dst) return;
    for (int i = 0; i < n; ++i) {
        size_t t = (size_t)c * LCH + i;
        memcpy(dst + (((size_t)b * J->T + t) * J->Nv + h) * width, src + (size_t)i * width, sizeof(double) * width);
    }
}

static void run_unit(const job_t *J, int b, int h, scratch_t *X)
{
    int d = J->d, dv = J->dv, T = J->T, P = J->Nv / 2, p = h / 2;
    int C = (T + LCH - 1) / LCH;
    size_t SS = (size_t)d * dv;
    double scale = 1.0 / sqrt((double)d);

    if (J->h0) memcpy(X->S, J->h0 + ((size_t)b * J->Nv + h) * SS, sizeof(double) * SS);
    else memset(X->S, 0, sizeof(double) * SS);

    double *orow = X->tmp; /* LCH x dv output rows */
    for (int c = 0; c < C; ++c) {
        int n = (c + 1) * LCH <= T ? LCH : T - c * LCH;
        int odd = c & 1;
        int sel = J->mask ? J->mask[((size_t)b * P + p) * C + c] != 0 : 1;
        if (!odd) memcpy(X->Sgrp, X->S, sizeof(double) * SS); /* group entry state S_c */
        if (J->s_in) memcpy(J->s_in + (((size_t)b * J->Nv + h) * C + c) * SS, X->S, sizeof(double) * SS);

        load_chunk(J, b, h, c, n, X->Qc, X->Kc, X->Vc, X->bet, X->gg);
        intra(J, n, X);
        if (J->score) {
            double acc = 0.0;
            int t0 = n > J->tail ? n - J->tail : 0;
            for (int t = t0; t < n; ++t)
                for (int j = 0; j < dv; ++j) acc += X->U[(size_t)t * dv + j] * X->U[(size_t)t * dv + j];
            J->score[((size_t)b * J->Nv + h) * C + c] = sqrt(acc);
        }
        if (J->cinv) memcpy(J->cinv + (((size_t)b * J->Nv + h) * C + c) * LCH * LCH, X->Cm, sizeof(double) * LCH * LCH);
        store_rows(J, J->u, b, h, c, n, X->U, dv);
        store_rows(J, J->w, b, h, c, n, X->W, d);

        /* the chunk form (Eqs. 3-4) reads the state entering this chunk */
        if (J->o_chunk) memcpy(X->Sent, X->S, sizeof(double) * SS);
        propagate(J, n, sel, X);
        store_rows(J, J->u_prime, b, h, c, n, X->Up, dv);
        if (J->o_chunk) {
            output_local(J, n, X->Qc, X->Kc, X->Up, X->gg, X->Sent, 0.0, orow);
            store_rows(J, J->o_chunk, b, h, c, n, orow, dv);
        }

        /* group-wise output (Eqs. 22-24) */
        if (!odd) {
            output_local(J, n, X->Qc, X->Kc, X->Up, X->gg, X->Sgrp, 0.0, orow);
            store_rows(J, J->o, b, h, c, n, orow, dv);
            /* remember chunk c for the odd chunk's cross term */
            memcpy(X->Qp, X->Qc, sizeof(double) * LCH * d);
            memcpy(X->Kp, X->Kc, sizeof(double) * LCH * d);
            memcpy(X->Up_prev, X->Up, sizeof(double) * LCH * dv);
            memcpy(X->gp, X->gg, sizeof(double) * LCH);
        } else {
            double gam_prev = X->gp[LCH - 1]; /* chunk c-1 is full whenever c is odd */
            output_local(J, n, X->Qc, X->Kc, X->Up, X->gg, X->Sgrp, gam_prev, orow);
            for (int i = 0; i < n; ++i)
                for (int s = 0; s < LCH; ++s) {
                    double a = dot(X->Qc + (size_t)i * d, X->Kp + (size_t)s * d, d)
                               * exp2(X->gg[i] + gam_prev - X->gp[s]) * scale;
                    for (int j = 0; j < dv; ++j) orow[(size_t)i * dv + j] += a * X->Up_prev[(size_t)s * dv + j];
                }
            store_rows(J, J->o, b, h, c, n, orow, dv);
        }
    }
    memcpy(J->s_final + ((size_t)b * J->Nv + h) * SS, X->S, sizeof(double) * SS);
}

typedef struct { const job_t *J; int tid; } worker_arg_t;

static void *worker(void *arg)
{
    const worker_arg_t *a = (const worker_arg_t *)arg;
    const job_t *J = a->J;
    int d = J->d, dv = J->dv;
    scratch_t X;
    size_t sz[] = {LCH * (size_t)d, LCH * (size_t)d, LCH * (size_t)dv, LCH, LCH,
                   LCH * LCH, LCH * LCH, LCH * (size_t)dv, LCH * (size_t)d, LCH * (size_t)dv,
                   LCH * (size_t)d, LCH * (size_t)d, LCH * (size_t)dv, LCH,
                   (size_t)d * dv, (size_t)d * dv, (size_t)d * dv, LCH * (size_t)dv};
    double **ptr[] = {&X.Qc, &X.Kc, &X.Vc, &X.bet, &X.gg, &X.M, &X.Cm, &X.U, &X.W, &X.Up,
                      &X.Qp, &X.Kp, &X.Up_prev, &X.gp, &X.S, &X.Sgrp, &X.Sent, &X.tmp};
    int nbuf = (int)(sizeof(sz) / sizeof(sz[0]));
    for (int i = 0; i < nbuf; ++i) *ptr[i] = (double *)calloc(sz[i], sizeof(double));
    int units = J->B * J->Nv;
    for (int u = a->tid; u < units; u += J->nthreads) run_unit(J, u / J->Nv, u % J->Nv, &X);
    for (int i = 0; i < nbuf; ++i) free(*ptr[i]);
    return NULL;
}

/* Full prefill.  All arrays are dense row-major fp64 (mask: uint8).
 *   q, k [B,T,Nq,d]; v [B,T,Nv,dv]; beta, g [B,T,Nv]; h0 [B,Nv,d,dv] or NULL;
 *   mask [B,Nv/2,ceil(T/64)] or NULL (= dense path, every chunk selected);
 *   o [B,T,Nv,dv]; s_final [B,Nv,d,dv].
 * Optional diagnostics (NULL to skip): o_chunk [B,T,Nv,dv] (chunk-form
 * output with the same states), u, u_prime [B,T,Nv,dv], w [B,T,Nv,d],
 * s_in [B,Nv,C,d,dv] (state entering each chunk), score [B,Nv,C],
 * cinv [B,Nv,C,64,64] (the solver's C).
 * Returns 0, or -1 on a bad argument. */
int gdn_oracle_prefill_tail(int B, int T, int Nq, int Nv, int d, int dv,
                            const double *q, const double *k, const double *v,
                            const double *beta, const double *g, const double *h0,
                            const unsigned char *mask, int solver, int nthreads,
                            double *o, double *s_final,
                            double *o_chunk, double *u, double *u_prime, double *w,
                            double *s_in, double *score, double *cinv, int tail)
{
    if (B < 0 || T < 0 || Nq <= 0 || Nv != 2 * Nq || d <= 0 || dv <= 0) return -1;
    if (solver != SOLVER_EXACT && solver != SOLVER_BLOCK_ADJ) return -1;
    if (tail < 1 || tail > LCH) return -1;
    if (!s_final || (T > 0 && (!q || !k || !v || !beta || !g || !o))) return -1;
    job_t J = {B, T, Nq, Nv, d, dv, solver, q, k, v, beta, g, h0, mask, o, s_final,
               o_chunk, u, u_prime, w, s_in, score, cinv, nthreads < 1 ? 1 : nthreads, tail};
    int units = B * Nv;
    if (J.nthreads > units) J.nthreads = units > 0 ? units : 1;
    pthread_t th[1024];
    worker_arg_t args[1024];
    if (J.nthreads > 1024) J.nthreads = 1024;
    for (int t = 0; t < J.nthreads; ++t) {
        args[t].J = &J; args[t].tid = t;
        pthread_create(&th[t], NULL, worker, &args[t]);
    }
    for (int t = 0; t < J.nthreads; ++t) pthread_join(th[t], NULL);
    return 0;
}

/* The prefill with the default Tail-16 score window. */
int gdn_oracle_prefill(int B, int T, int Nq, int Nv, int d, int dv,
                       const double *q, const double *k, const double *v,
                       const double *beta, const double *g, const double *h0,
                       const unsigned char *mask, int solver, int nthreads,
                       double *o, double *s_final,
                       double *o_chunk, double *u, double *u_prime, double *w,
                       double *s_in, double *score, double *cinv)
{
    return gdn_oracle_prefill_tail(B, T, Nq, Nv, d, dv, q, k, v, beta, g, h0, mask, solver, nthreads, o, s_final,
                                   o_chunk, u, u_prime, w, s_in, score, cinv, BLK);
}

/* ---- event compaction (Sec. 2.5 CSR layout) ------------------------------
 * Rows: one per (sequence b, head pair p), physical id i = b*P + p, ordered by
 * event count descending, ties by physical id ascending (a caller mask has no
 * tiers; "long chains first").  Events inside a row ascend in chunk index.
 *   row_pair[j]      physical id of row j                           [B*P]
 *   row_ptr[j]       offset of row j's first event; row_ptr[B*P] = E [B*P+1]
 *   ev_chunk[e]      chunk index of event e                         [E]
 *   grp_pred[i*G+r]  global index of the last event of pair i with chunk < 2r,
 *                    or -1 (G = ceil(C/2))                          [B*P*G]
 *   snap_slot[e]     dense number, in global event order, of the events that
 *                    are some group's predecessor; -1 otherwise     [E]
 * Returns 0, 1 when E exceeds `capacity` (outputs beyond row_ptr untouched),
 * -1 on a bad argument. */
int gdn_oracle_events(int B, int P, int C, const unsigned char *mask, int capacity,
                      int *row_pair, int *row_ptr, int *ev_chunk, int *grp_pred,
                      int *snap_slot, int *n_events, int *n_snap)
{
    if (B < 0 || P <= 0 || C < 0) return -1;
    int R = B * P, G = (C + 1) / 2;
    int *cnt = (int *)calloc(R > 0 ? R : 1, sizeof(int));
    for (int i = 0; i < R; ++i)
        for (int c = 0; c < C; ++c) cnt[i] += mask[(size_t)i * C + c] != 0;
    /* insertion sort: count descending, id ascending */
    for (int i = 0; i < R; ++i) row_pair[i] = i;
    for (int i = 1; i < R; ++i) {
        int x = row_pair[i], j = i - 1;
        while (j >= 0 && (cnt[row_pair[j]] < cnt[x] || (cnt[row_pair[j]] == cnt[x] && row_pair[j] > x))) {
            row_pair[j + 1] = row_pair[j];
            --j;
        }
        row_pair[j + 1] = x;
    }
    row_ptr[0] = 0;
    for (int j = 0; j < R; ++j) row_ptr[j + 1] = row_ptr[j] + cnt[row_pair[j]];
    int E = row_ptr[R];
    *n_events = E;
    if (E > capacity) { free(cnt); *n_snap = 0; return 1; }
    for (int j = 0; j < R; ++j) {
        int i = row_pair[j], e = row_ptr[j];
        for (int c = 0; c < C; ++c)
            if (mask[(size_t)i * C + c]) ev_chunk[e++] = c;
    }
    for (int e = 0; e < E; ++e) snap_slot[e] = -1;
    for (int j = 0; j < R; ++j) {
        int i = row_pair[j];
        for (int r = 0; r < G; ++r) {
            int pred = -1;
            for (int e = row_ptr[j]; e < row_ptr[j + 1]; ++e)
                if (ev_chunk[e] < 2 * r) pred = e;
            grp_pred[(size_t)i * G + r] = pred;
            if (pred >= 0) snap_slot[pred] = -2; /* mark: referenced by a group */
        }
    }
    int ns = 0;
    for (int e = 0; e < E; ++e)
        if (snap_slot[e] == -2) snap_slot[e] = ns++;
    *n_snap = ns;
    free(cnt);
    return 0;
}

/* ---- online event selection (Sec. 2.4, Eqs. 10-14) -----------------------
 * Per sequence, from the Tail-16 scores s[h][c] (Eq. 9), the chunk gate tails
 * gamma[h][c] and an optional output-visibility energy eta[h]:
 *   norm_h = ||s_{.,h}||_2 (sum of squares in fp64, rounded to fp32, fp32 sqrt)
 *   q_c    = 0.5 (s_{c,h0} / norm_h0 + s_{c,h1} / norm_h1), fp32 (Eq. 10); a zero norm adds 0
 *   r_h    = mean of 2^gamma over the last min(16, C) chunks; L_h = sum_{j=1}^{C-2} r_h^j (Eq. 11)
 *   G_h    = sqrt(eta_h / mean eta), or 1 without eta (Eq. 11)
 *   k_l    = clip(round_half_even(rho_l C), 2, C), rho = (0.08, 0.30, 0.95); C = 1 keeps its chunk
 *   C_l    = anchors {0, C-1} plus the k_l - 2 best non-anchor chunks by q (ties: lower index)
 *            -- nested sets C_L in C_M in C_H (Eq. 13)
 *   gains  Delta_{a->b} = sum_{c in C_b \ C_a} sum_{h in pair} s_{c,h} L_h G_h (Eq. 12), fp64
 *   x      = gains / mean over pairs (0 when the mean is 0)
 *   B(x,k) = k (n-k) / n (mean of the k largest - mean of the rest)^2 (Eq. 14)
 *   n_H    = argmax_{k in 1..4} B(x_H sorted desc, k), n = 16 (ties: smaller k); the n_H pairs
 *            with the largest x_H (ties: lower pair id) take tier H
 *   n_M    = argmax over the row {1: 11-13, 2: 7-9, 3: 3-5, 4: 0} of B(x_M of the other pairs), n = 16 - n_H;
 *            the n_M best of the other pairs by x_M take tier M; the rest tier L.
 *   mask[p][c] = [c in C_tier(p)], shared by the pair.
 * Only defined for 16 head pairs (the pages' tier table).  Returns 0, or -1. */
typedef struct { float q; int c; } ranked_t;

/* q descending, ties: lower chunk index first */
static int cmp_ranked(const void *a, const void *b)
{
    const ranked_t *x = (const ranked_t *)a, *y = (const ranked_t *)b;
    if (x->q != y->q) return x->q > y->q ? -1 : 1;
    return x->c < y->c ? -1 : (x->c > y->c);
}

/* B(x, k) for x sorted descending (Eq. 14) */
static double separation(const double *xs, int n, int k)
{
    double top = 0.0, rest = 0.0;
    for (int i = 0; i < k; ++i) top += xs[i];
    for (int i = k; i < n; ++i) rest += xs[i];
    top /= k;
    rest = n > k ? rest / (n - k) : 0.0;
    return (double)k * (n - k) / n * (top - rest) * (top - rest);
}

/* sort pair ids by x descending, ties: lower id first (insertion sort, n <= 16) */
static void order_pairs(const double *x, int *ids, int n)
{
    for (int i = 1; i < n; ++i) {
        int v = ids[i], j = i - 1;
        while (j >= 0 && (x[ids[j]] < x[v] || (x[ids[j]] == x[v] && ids[j] > v))) {
            ids[j + 1] = ids[j];
            --j;
        }
        ids[j + 1] = v;
    }
}

int gdn_oracle_select(int B, int Nv, int C, const float *score, const float *gamma, const float *eta,
                      unsigned char *mask, int *tier_out, int *k_out)
{
    enum { NP = 16 };
    if (Nv != 2 * NP || C < 0 || B < 0) return -1;
    const double rho[3] = {0.08, 0.30, 0.95};       /* tiers L, M, H */
    static const int nm_lo[5] = {0, 11, 7, 3, 0}, nm_hi[5] = {0, 13, 9, 5, 0};
    int k[3];
    for (int l = 0; l < 3; ++l) {
        int kk = (int)nearbyint(rho[l] * C);          /* round half to even */
        kk = kk < 2 ? 2 : kk;
        k[l] = kk > C ? C : kk;
    }
    if (k_out) for (int l = 0; l < 3; ++l) k_out[l] = k[l];
    const int n_in = C > 2 ? C - 2 : 0;               /* non-anchor chunks 1 .. C-2 */
    ranked_t *rk = (ranked_t *)malloc(sizeof(ranked_t) * (n_in > 0 ? n_in : 1));
    int *rank = (int *)malloc(sizeof(int) * (size_t)NP * (C > 0 ? C : 1));  /* -1: anchor */

    for (int b = 0; b < B; ++b) {
        const float *s = score + (size_t)b * Nv * C;  /* s[h * C + c] */
        const float *gm = gamma + (size_t)b * Nv * C;
        float norm[2 * NP];
        double L[2 * NP], G[2 * NP];
        /* Eq. 11: norms, memory lifetime, output visibility */
        for (int h = 0; h < Nv; ++h) {
            double ss = 0.0;
            for (int c = 0; c < C; ++c) ss += (double)s[h * C + c] * (double)s[h * C + c];
            norm[h] = sqrtf((float)ss);
            const int c0 = C > 16 ? C - 16 : 0;
            double r = 0.0;
            for (int c = c0; c < C; ++c) r += exp2((double)gm[h * C + c]);
            r = C > c0 ? r / (C - c0) : 0.0;
            double Lh = 0.0, pw = 1.0;
            for (int j = 1; j <= C - 2; ++j) { pw *= r; Lh += pw; }
            L[h] = Lh;
        }
        double emean = 0.0;
        if (eta) {
            for (int h = 0; h < Nv; ++h) emean += eta[(size_t)b * Nv + h];
            emean /= Nv;
        }
        for (int h = 0; h < Nv; ++h)
            G[h] = !eta ? 1.0 : (emean > 0.0 ? sqrt(eta[(size_t)b * Nv + h] / emean) : 0.0);

        /* Eqs. 10, 12, 13: in-pair ranking, nested candidate sets, upgrade gains */
        double gain_LM[NP], gain_MH[NP];
        for (int p = 0; p < NP; ++p) {
            const int h0 = 2 * p, h1 = 2 * p + 1;
            for (int i = 0; i < n_in; ++i) {
                const int c = i + 1;
                const float a0 = norm[h0] > 0.f ? s[h0 * C + c] / norm[h0] : 0.f;
                const float a1 = norm[h1] > 0.f ? s[h1 * C + c] / norm[h1] : 0.f;
                rk[i].q = 0.5f * (a0 + a1);
                rk[i].c = c;
            }
            qsort(rk, n_in, sizeof(ranked_t), cmp_ranked);
            int *rp = rank + (size_t)p * C;
            for (int c = 0; c < C; ++c) rp[c] = -1;
            for (int i = 0; i < n_in; ++i) rp[rk[i].c] = i;
            gain_LM[p] = gain_MH[p] = 0.0;
            for (int i = 0; i < n_in; ++i) {
                const int c = rk[i].c;
                const double w = (double)s[h0 * C + c] * L[h0] * G[h0] + (double)s[h1 * C + c] * L[h1] * G[h1];
                if (i >= k[0] - 2 && i < k[1] - 2) gain_LM[p] += w;   /* in C_M, not in C_L */
                if (i >= k[1] - 2 && i < k[2] - 2) gain_MH[p] += w;   /* in C_H, not in C_M */
            }
        }

        /* Eq. 14: dynamic tier counts */
        double mLM = 0.0, mMH = 0.0, xM[NP], xH[NP], xs[NP];
        for (int p = 0; p < NP; ++p) { mLM += gain_LM[p]; mMH += gain_MH[p]; }
        mLM /= NP;
        mMH /= NP;
        for (int p = 0; p < NP; ++p) {
            xM[p] = mLM != 0.0 ? gain_LM[p] / mLM : 0.0;
            xH[p] = mMH != 0.0 ? gain_MH[p] / mMH : 0.0;
        }
        int ids[NP], tier[NP];
        for (int p = 0; p < NP; ++p) { ids[p] = p; tier[p] = 0; }
        order_pairs(xH, ids, NP);
        for (int i = 0; i < NP; ++i) xs[i] = xH[ids[i]];
        int nH = 1;
        double best = separation(xs, NP, 1);
        for (int kk = 2; kk <= 4; ++kk) {
            const double v = separation(xs, NP, kk);
            if (v > best) { best = v; nH = kk; }
        }
        for (int i = 0; i < nH; ++i) tier[ids[i]] = 2;
        int rest[NP], nr = 0;
        for (int p = 0; p < NP; ++p)
            if (tier[p] != 2) rest[nr++] = p;
        order_pairs(xM, rest, nr);
        for (int i = 0; i < nr; ++i) xs[i] = xM[rest[i]];
        int nM = 0;
        if (nm_hi[nH] > 0) {
            nM = nm_lo[nH];
            best = separation(xs, nr, nM);
            for (int kk = nm_lo[nH] + 1; kk <= nm_hi[nH]; ++kk) {
                const double v = separation(xs, nr, kk);
                if (v > best) { best = v; nM = kk; }
            }
        }
        for (int i = 0; i < nM; ++i) tier[rest[i]] = 1;

        /* the mask of each pair: anchors plus its tier's best k - 2 chunks */
        for (int p = 0; p < NP; ++p) {
            if (tier_out) tier_out[(size_t)b * NP + p] = tier[p];
            const int *rp = rank + (size_t)p * C;
            for (int c = 0; c < C; ++c)
                mask[((size_t)b * NP + p) * C + c] = (rp[c] < 0 || rp[c] < k[tier[p]] - 2) ? 1 : 0;
        }
    }
    free(rk);
    free(rank);
    return 0;
}

/* One decode step for B sequences (Eqs. 1-4 with L = 1; see the header).
 * q, k [B, Nq, d]; v [B, Nv, dv]; beta, a [B, Nv]; S [B, Nv, d, dv] updated in
 * place; o [B, Nv, dv].  Value head h reads query/key head h / 2. */
int gdn_oracle_decode(int B, int Nq, int Nv, int d, int dv, const double *q, const double *k, const double *v,
                      const double *beta, const double *a, double *S, double *o)
{
    if (B < 0 || Nq <= 0 || Nv != 2 * Nq || d <= 0 || dv <= 0) return -1;
    double *wS = (double *)malloc(sizeof(double) * (size_t)dv);
    double *up = (double *)malloc(sizeof(double) * (size_t)dv);
    double *qS = (double *)malloc(sizeof(double) * (size_t)dv);
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Nv; ++h) {
            const int p = h / 2;
            const double *qt = q + ((size_t)b * Nq + p) * d, *kt = k + ((size_t)b * Nq + p) * d;
            const double *vt = v + ((size_t)b * Nv + h) * dv;
            const double bt = beta[(size_t)b * Nv + h], at = a[(size_t)b * Nv + h];
            double *Sh = S + ((size_t)b * Nv + h) * d * dv;
            const double decay = pow(2.0, at), qk = dot(qt, kt, d);
            for (int j = 0; j < dv; ++j) {          /* W S = beta 2^a (k^T S), and q^T S */
                double ks = 0.0, qs = 0.0;
                for (int i = 0; i < d; ++i) {
                    ks += kt[i] * Sh[(size_t)i * dv + j];
                    qs += qt[i] * Sh[(size_t)i * dv + j];
                }
                wS[j] = bt * decay * ks;
                qS[j] = qs;
            }
            for (int j = 0; j < dv; ++j) up[j] = bt * vt[j] - wS[j];   /* U' = U - W S */
            for (int i = 0; i < d; ++i)                                /* S+ = 2^a S + k U'^T */
                for (int j = 0; j < dv; ++j)
                    Sh[(size_t)i * dv + j] = decay * Sh[(size_t)i * dv + j] + kt[i] * up[j];
            for (int j = 0; j < dv; ++j)
                o[((size_t)b * Nv + h) * dv + j] = (decay * qS[j] + qk * up[j]) / sqrt((double)d);
        }
    free(wS);
    free(up);
    free(qS);
    return 0;
}
