/*
 * CPU oracle of the sparse-delta-memory (SDM) write/read: plain, slow, fp64.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker of the CUDA path, not part of it:
 * only the test-suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Source of every definition: the sparse-delta-memory 2.0.0 wheel pages,
 *   - memory_ops.py, module docstring ("Forward: Phase 1 / solve / Phase 2") and the
 *     SDMWriteRead docstring (the reference token loop);
 *   - phase2_kernels.py, module docstring (layout, padding, determinism and the sorted
 *     "kind row" groups) and the _sdm_dual_matmul docstring;
 *   - wy_solve.py, module docstring (X = (I + L)^-1, QX = QK X).
 *
 * Layout (all row-major, per stream p of P):
 *   bank   [P*S, D]   stream p owns rows [p*S, (p+1)*S); slot ids are per stream, 0..S-1
 *   ws, k, g [P, T, W]  write slots, write weights, log-decays (one per write entry)
 *   beta   [P, T]
 *   v      [P, T, D]
 *   rs, q  [P, T, R]  read slots, read weights
 *   valid  [P]        tokens t >= valid[p] are padding: no bank access, zero readings
 *   out    [P, T, D]  readings
 *
 * Return codes: 0 ok, -1 invalid argument (slot out of range, repeated write slot in a
 * token, bad sizes), -2 out of memory.
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
#define ORACLE_ENOMEM (-2)

static int check_sizes(int P, int T, int S, int D, int W, int R) {
    return (P >= 1 && T >= 1 && S >= 1 && D >= 1 && W >= 1 && R >= 1) ? ORACLE_OK : ORACLE_EINVAL;
}

/* Slots of one token: all in [0, S); write slots pairwise distinct (a precondition of the
 * op, memory_ops.py sdm_write_read docstring: "the W slots of a token must be distinct"). */
static int check_token(const int32_t *ws, int W, const int32_t *rs, int R, int S) {
    for (int j = 0; j < W; ++j) {
        if (ws[j] < 0 || ws[j] >= S) return ORACLE_EINVAL;
        for (int jj = 0; jj < j; ++jj)
            if (ws[jj] == ws[j]) return ORACLE_EINVAL;
    }
    for (int i = 0; i < R; ++i)
        if (rs[i] < 0 || rs[i] >= S) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------
 * The reference token loop (memory_ops.py, SDMWriteRead docstring), one stream:
 *   a_j   = B[s_j]                     the rows the token writes, before it writes
 *   d_j   = exp(g_j) * a_j             only the written rows decay
 *   ret   = sum_j k_j * d_j            retrieved
 *   u     = beta * (v - ret)           delta_v
 *   B[s_j] = d_j + k_j * u             (bank[k] += read - at_k + k_val (x) delta_v)
 *   o     = sum_i q_i * B[r_i]         readings, after the write
 * ------------------------------------------------------------------------------------ */
static int sequential_stream(int T, int S, int D, int W, int R, double *B, const int32_t *ws,
                             const double *k, const double *g, const double *beta,
                             const double *v, const int32_t *rs, const double *q, int valid,
                             double *out, double *a /* [W*D] */, double *ret /* [D] */,
                             double *a_log /* [T*W*D] or NULL */) {
    (void)S;
    for (int t = 0; t < T; ++t) {
        double *o = out + (size_t)t * D;
        if (t >= valid) {
            memset(o, 0, sizeof(double) * D);
            continue;
        }
        const int32_t *s = ws + (size_t)t * W;
        const int32_t *r = rs + (size_t)t * R;
        const double *kt = k + (size_t)t * W, *gt = g + (size_t)t * W, *qt = q + (size_t)t * R;
        const double *vt = v + (size_t)t * D;
        int rc = check_token(s, W, r, R, S);
        if (rc) return rc;
        /* a_j, then d_j in place */
        for (int j = 0; j < W; ++j) {
            memcpy(a + (size_t)j * D, B + (size_t)s[j] * D, sizeof(double) * D);
            if (a_log) memcpy(a_log + ((size_t)t * W + j) * D, a + (size_t)j * D, sizeof(double) * D);
        }
        for (int j = 0; j < W; ++j) {
            double e = exp(gt[j]);
            for (int c = 0; c < D; ++c) a[(size_t)j * D + c] *= e;
        }
        for (int c = 0; c < D; ++c) ret[c] = 0.0;
        for (int j = 0; j < W; ++j)
            for (int c = 0; c < D; ++c) ret[c] += kt[j] * a[(size_t)j * D + c];
        /* u overwrites ret */
        for (int c = 0; c < D; ++c) ret[c] = beta[t] * (vt[c] - ret[c]);
        for (int j = 0; j < W; ++j) {
            double *row = B + (size_t)s[j] * D;
            for (int c = 0; c < D; ++c) row[c] = a[(size_t)j * D + c] + kt[j] * ret[c];
        }
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        for (int i = 0; i < R; ++i) {
            const double *row = B + (size_t)r[i] * D;
            for (int c = 0; c < D; ++c) o[c] += qt[i] * row[c];
        }
    }
    return ORACLE_OK;
}

/* Sequential recurrence over all P streams (streams own disjoint rows, so they are
 * independent; nthreads > 1 runs them on OpenMP threads). bank is advanced in place. */
int sdm_oracle_sequential(int P, int T, int S, int D, int W, int R, double *bank,
                          const int32_t *ws, const double *k, const double *g,
                          const double *beta, const double *v, const int32_t *rs,
                          const double *q, const int32_t *valid, double *out, int nthreads) {
    if (check_sizes(P, T, S, D, W, R)) return ORACLE_EINVAL;
    for (int p = 0; p < P; ++p)
        if (valid[p] < 0 || valid[p] > T) return ORACLE_EINVAL;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int p = 0; p < P; ++p) {
        double *a = (double *)malloc(sizeof(double) * ((size_t)W * D + D));
        int rc;
        if (!a) {
            rc = ORACLE_ENOMEM;
        } else {
            rc = sequential_stream(T, S, D, W, R, bank + (size_t)p * S * D,
                                   ws + (size_t)p * T * W, k + (size_t)p * T * W,
                                   g + (size_t)p * T * W, beta + (size_t)p * T,
                                   v + (size_t)p * T * D, rs + (size_t)p * T * R,
                                   q + (size_t)p * T * R, valid[p], out + (size_t)p * T * D, a,
                                   a + (size_t)W * D, NULL);
        }
        free(a);
        if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------------------
 * The chunked form (memory_ops.py module docstring; phase2_kernels.py module docstring;
 * wy_solve.py module docstring), written from the definitions, in fp64, one chunk of one
 * stream at a time. Chunk c covers tokens c*C .. c*C+C-1; n = number of valid ones.
 *
 * Phase 1 (memory-independent, per chunk):
 *   lam(s, t)   running sum of g over the writes of slot s at tokens <= t of the chunk
 *   Lw[t][j]    = lam(s_tj, t)            (inclusive: the token's own decay)
 *   Lr[t][i]    = lam(r_ti, t)            (0 if the chunk has not written r_ti by t)
 *   Lend(s)     = lam(s, last token)
 *   gw[t][j]    = k_tj * exp(Lw[t][j])     gather weight of a write entry
 *   qw[t][i]    = q_ti * exp(Lr[t][i])     gather weight of a read entry
 *   dw[t][j]    = k_tj * exp(Lend(s_tj) - Lw[t][j])   write weight of the DW
 *   A[t][u]     = sum_{j,j': s_tj = s_uj'} k_tj k_uj' exp(Lw[t][j] - Lw[u][j'])   u < t
 *   QK[t][u]    = sum_{i,j': r_ti = s_uj'} q_ti k_uj' exp(Lr[t][i] - Lw[u][j'])  u <= t
 * Solve:  X = (I + tril(diag(beta) A, -1))^-1 ;  QX = QK X
 * Phase 2 (with B0 = the bank at the chunk start):
 *   retrieved[t] = sum_j gw[t][j] B0[s_tj] ;  inter[t] = sum_i qw[t][i] B0[r_ti]
 *   u_pre[t] = beta_t (v_t - retrieved[t]) ;  delta_v = X u_pre ;  readings = QX u_pre + inter
 *   DW: B[s] = exp(Lend(s)) B0[s] + sum_{(t,j): s_tj = s} dw[t][j] delta_v[t]
 * ------------------------------------------------------------------------------------ */

typedef struct {
    int C, D, W, R, n;        /* n valid tokens in the chunk */
    double *Lw, *Lr, *gw, *qw, *dw;   /* [C*W], [C*R] */
    double *A, *QK, *X, *QX;          /* [C*C] */
    double *ret, *inter, *upre, *dv, *rd;  /* [C*D] */
    double *lam;                      /* [S] running sums, all zero between chunks */
    unsigned char *touched;           /* [S] */
    double *lend;                     /* [C*W] Lend(s_tj) per write entry */
} chunk_ws;

static void chunk_phase1(chunk_ws *c, const int32_t *ws, const double *k, const double *g,
                         const int32_t *rs, const double *q) {
    const int W = c->W, R = c->R, n = c->n, C = c->C;
    /* running sums in token order */
    for (int t = 0; t < n; ++t) {
        for (int j = 0; j < W; ++j) {
            int s = ws[t * W + j];
            c->lam[s] += g[t * W + j];
            c->touched[s] = 1;
            c->Lw[t * W + j] = c->lam[s];
        }
        for (int i = 0; i < R; ++i) c->Lr[t * R + i] = c->lam[rs[t * R + i]];
    }
    for (int t = 0; t < n; ++t)
        for (int j = 0; j < W; ++j) c->lend[t * W + j] = c->lam[ws[t * W + j]];
    /* reset the running sums of the touched slots */
    for (int t = 0; t < n; ++t)
        for (int j = 0; j < W; ++j) {
            int s = ws[t * W + j];
            c->lam[s] = 0.0;
            c->touched[s] = 0;
        }
    for (int t = 0; t < n; ++t) {
        for (int j = 0; j < W; ++j) {
            double kk = k[t * W + j], lw = c->Lw[t * W + j];
            c->gw[t * W + j] = kk * exp(lw);
            c->dw[t * W + j] = kk * exp(c->lend[t * W + j] - lw);
        }
        for (int i = 0; i < R; ++i) c->qw[t * R + i] = q[t * R + i] * exp(c->Lr[t * R + i]);
    }
    memset(c->A, 0, sizeof(double) * C * C);
    memset(c->QK, 0, sizeof(double) * C * C);
    for (int t = 0; t < n; ++t)
        for (int u = 0; u <= t; ++u) {
            double a = 0.0, qk = 0.0;
            for (int jp = 0; jp < W; ++jp) {
                int su = ws[u * W + jp];
                double ku = k[u * W + jp], lu = c->Lw[u * W + jp];
                if (u < t)
                    for (int j = 0; j < W; ++j)
                        if (ws[t * W + j] == su) a += k[t * W + j] * ku * exp(c->Lw[t * W + j] - lu);
                for (int i = 0; i < R; ++i)
                    if (rs[t * R + i] == su) qk += q[t * R + i] * ku * exp(c->Lr[t * R + i] - lu);
            }
            c->A[t * C + u] = a;
            c->QK[t * C + u] = qk;
        }
}

/* X = (I + L)^-1 with L = tril(diag(beta) A, -1), by forward substitution row by row:
 * X[t][:] = e_t - sum_{u<t} L[t][u] X[u][:]. Padding rows (t >= n) are identity rows. */
static void chunk_solve(chunk_ws *c, const double *beta) {
    const int C = c->C;
    for (int t = 0; t < C; ++t) {
        double *xt = c->X + (size_t)t * C;
        for (int col = 0; col < C; ++col) xt[col] = (col == t) ? 1.0 : 0.0;
        if (t >= c->n) continue;
        for (int u = 0; u < t; ++u) {
            double l = beta[t] * c->A[t * C + u];
            if (l == 0.0) continue;
            const double *xu = c->X + (size_t)u * C;
            for (int col = 0; col <= u; ++col) xt[col] -= l * xu[col];
        }
    }
    for (int t = 0; t < C; ++t)
        for (int col = 0; col < C; ++col) {
            double s = 0.0;
            for (int u = 0; u <= t; ++u) s += c->QK[t * C + u] * c->X[u * C + col];
            c->QX[t * C + col] = s;
        }
}

static void chunk_phase2(chunk_ws *c, double *B, const int32_t *ws, const int32_t *rs,
                         const double *beta, const double *v, double *out) {
    const int C = c->C, D = c->D, W = c->W, R = c->R, n = c->n;
    memset(c->ret, 0, sizeof(double) * C * D);
    memset(c->inter, 0, sizeof(double) * C * D);
    for (int t = 0; t < n; ++t) {
        for (int j = 0; j < W; ++j) {
            const double *row = B + (size_t)ws[t * W + j] * D;
            for (int d = 0; d < D; ++d) c->ret[t * D + d] += c->gw[t * W + j] * row[d];
        }
        for (int i = 0; i < R; ++i) {
            const double *row = B + (size_t)rs[t * R + i] * D;
            for (int d = 0; d < D; ++d) c->inter[t * D + d] += c->qw[t * R + i] * row[d];
        }
    }
    for (int t = 0; t < C; ++t)
        for (int d = 0; d < D; ++d)
            c->upre[t * D + d] = t < n ? beta[t] * (v[t * D + d] - c->ret[t * D + d]) : 0.0;
    for (int t = 0; t < C; ++t)
        for (int d = 0; d < D; ++d) {
            double a = 0.0, b = 0.0;
            for (int u = 0; u < C; ++u) {
                a += c->X[t * C + u] * c->upre[u * D + d];
                b += c->QX[t * C + u] * c->upre[u * D + d];
            }
            c->dv[t * D + d] = t < n ? a : 0.0;
            c->rd[t * D + d] = t < n ? b + c->inter[t * D + d] : 0.0;
        }
    for (int t = 0; t < n; ++t) memcpy(out + (size_t)t * D, c->rd + (size_t)t * D, sizeof(double) * D);
    /* DW: every written slot once, from B0 (first occurrence in the chunk decides). */
    for (int t = 0; t < n; ++t)
        for (int j = 0; j < W; ++j) {
            int s = ws[t * W + j];
            int first = 1;
            for (int u = 0; u < t && first; ++u)
                for (int jp = 0; jp < W; ++jp)
                    if (ws[u * W + jp] == s) { first = 0; break; }
            if (!first) continue;
            double *row = B + (size_t)s * D;
            double f = exp(c->lend[t * W + j]);
            for (int d = 0; d < D; ++d) row[d] *= f;
            for (int u = t; u < n; ++u)
                for (int jp = 0; jp < W; ++jp)
                    if (ws[u * W + jp] == s)
                        for (int d = 0; d < D; ++d) row[d] += c->dw[u * W + jp] * c->dv[u * D + d];
        }
}

static void chunk_ws_free(chunk_ws *c) {
    free(c->Lw); free(c->Lr); free(c->gw); free(c->qw); free(c->dw); free(c->lend);
    free(c->A); free(c->QK); free(c->X); free(c->QX);
    free(c->ret); free(c->inter); free(c->upre); free(c->dv); free(c->rd);
    free(c->lam); free(c->touched);
}

static int chunk_ws_alloc(chunk_ws *c, int C, int S, int D, int W, int R) {
    memset(c, 0, sizeof(*c));
    c->C = C; c->D = D; c->W = W; c->R = R;
    size_t cw = (size_t)C * W, cr = (size_t)C * R, cc = (size_t)C * C, cd = (size_t)C * D;
    c->Lw = calloc(cw, sizeof(double)); c->gw = calloc(cw, sizeof(double));
    c->dw = calloc(cw, sizeof(double)); c->lend = calloc(cw, sizeof(double));
    c->Lr = calloc(cr, sizeof(double)); c->qw = calloc(cr, sizeof(double));
    c->A = calloc(cc, sizeof(double)); c->QK = calloc(cc, sizeof(double));
    c->X = calloc(cc, sizeof(double)); c->QX = calloc(cc, sizeof(double));
    c->ret = calloc(cd, sizeof(double)); c->inter = calloc(cd, sizeof(double));
    c->upre = calloc(cd, sizeof(double)); c->dv = calloc(cd, sizeof(double));
    c->rd = calloc(cd, sizeof(double));
    c->lam = calloc((size_t)S, sizeof(double));
    c->touched = calloc((size_t)S, 1);
    if (!c->Lw || !c->gw || !c->dw || !c->lend || !c->Lr || !c->qw || !c->A || !c->QK || !c->X ||
        !c->QX || !c->ret || !c->inter || !c->upre || !c->dv || !c->rd || !c->lam || !c->touched) {
        chunk_ws_free(c);
        return ORACLE_ENOMEM;
    }
    return ORACLE_OK;
}

/* Chunked form over all streams; bank advanced in place; readings to out.
 * dbg_*: when non-NULL, the intermediates of chunk (dbg_p, dbg_chunk) are copied out:
 *   dbg_lw [C*W], dbg_lr [C*R], dbg_gw [C*W], dbg_qw [C*R], dbg_dw [C*W],
 *   dbg_A, dbg_QK, dbg_X, dbg_QX [C*C], dbg_ret, dbg_inter, dbg_dv [C*D]. */
int sdm_oracle_chunked(int P, int T, int C, int S, int D, int W, int R, double *bank,
                       const int32_t *ws, const double *k, const double *g, const double *beta,
                       const double *v, const int32_t *rs, const double *q,
                       const int32_t *valid, double *out, int dbg_p, int dbg_chunk,
                       double *dbg_lw, double *dbg_lr, double *dbg_gw, double *dbg_qw,
                       double *dbg_dw, double *dbg_A, double *dbg_QK, double *dbg_X,
                       double *dbg_QX, double *dbg_ret, double *dbg_inter, double *dbg_dv) {
    if (check_sizes(P, T, S, D, W, R) || C < 1) return ORACLE_EINVAL;
    chunk_ws c;
    if (chunk_ws_alloc(&c, C, S, D, W, R)) return ORACLE_ENOMEM;
    int rc = ORACLE_OK;
    memset(out, 0, sizeof(double) * (size_t)P * T * D);
    for (int p = 0; p < P && !rc; ++p) {
        if (valid[p] < 0 || valid[p] > T) { rc = ORACLE_EINVAL; break; }
        double *B = bank + (size_t)p * S * D;
        int nt = (T + C - 1) / C;
        for (int ci = 0; ci < nt && !rc; ++ci) {
            int t0 = ci * C;
            int n = valid[p] - t0;
            if (n < 0) n = 0;
            if (n > C) n = C;
            c.n = n;
            const int32_t *cws = ws + ((size_t)p * T + t0) * W;
            const int32_t *crs = rs + ((size_t)p * T + t0) * R;
            for (int t = 0; t < n && !rc; ++t)
                rc = check_token(cws + (size_t)t * W, W, crs + (size_t)t * R, R, S);
            if (rc) break;
            const double *ck = k + ((size_t)p * T + t0) * W, *cg = g + ((size_t)p * T + t0) * W;
            const double *cq = q + ((size_t)p * T + t0) * R;
            const double *cb = beta + (size_t)p * T + t0, *cv = v + ((size_t)p * T + t0) * D;
            chunk_phase1(&c, cws, ck, cg, crs, cq);
            chunk_solve(&c, cb);
            chunk_phase2(&c, B, cws, crs, cb, cv, out + ((size_t)p * T + t0) * D);
            if (p == dbg_p && ci == dbg_chunk) {
                size_t cw = (size_t)C * W, cr = (size_t)C * R, cc = (size_t)C * C, cd = (size_t)C * D;
                if (dbg_lw) memcpy(dbg_lw, c.Lw, cw * sizeof(double));
                if (dbg_lr) memcpy(dbg_lr, c.Lr, cr * sizeof(double));
                if (dbg_gw) memcpy(dbg_gw, c.gw, cw * sizeof(double));
                if (dbg_qw) memcpy(dbg_qw, c.qw, cr * sizeof(double));
                if (dbg_dw) memcpy(dbg_dw, c.dw, cw * sizeof(double));
                if (dbg_A) memcpy(dbg_A, c.A, cc * sizeof(double));
                if (dbg_QK) memcpy(dbg_QK, c.QK, cc * sizeof(double));
                if (dbg_X) memcpy(dbg_X, c.X, cc * sizeof(double));
                if (dbg_QX) memcpy(dbg_QX, c.QX, cc * sizeof(double));
                if (dbg_ret) memcpy(dbg_ret, c.ret, cd * sizeof(double));
                if (dbg_inter) memcpy(dbg_inter, c.inter, cd * sizeof(double));
                if (dbg_dv) memcpy(dbg_dv, c.dv, cd * sizeof(double));
            }
            /* entries of the chunk that were never valid leave Lw etc. from an earlier
             * chunk in place; clear them so a later debug copy shows zeros there */
            memset(c.Lw, 0, sizeof(double) * C * W); memset(c.gw, 0, sizeof(double) * C * W);
            memset(c.dw, 0, sizeof(double) * C * W); memset(c.lend, 0, sizeof(double) * C * W);
            memset(c.Lr, 0, sizeof(double) * C * R); memset(c.qw, 0, sizeof(double) * C * R);
        }
    }
    chunk_ws_free(&c);
    return rc;
}

/* ------------------------------------------------------------------------------------
 * The dedup plan of one chunk (phase2_kernels.py module docstring, "Determinism"):
 * the entries of a kind (writes: e = t*W + j; reads: e = t*R + i) sorted by (slot, e)
 * form the kind row; a group is a maximal run of one slot; an entry whose slot occurs once
 * is "only"; the group's owner is its last entry. Only the n valid tokens take part.
 * Outputs (m = n * width entries): perm[m] (entry index at each sorted position),
 * group_start[m] (1 where a group begins), owner[m] (1 at a group's last entry),
 * only[m] (1 where the group has one entry). Returns the number of groups.
 * ------------------------------------------------------------------------------------ */
typedef struct { int32_t slot; int32_t e; } plan_key;

static int plan_cmp(const void *x, const void *y) {
    const plan_key *a = (const plan_key *)x, *b = (const plan_key *)y;
    if (a->slot != b->slot) return a->slot < b->slot ? -1 : 1;
    return (a->e > b->e) - (a->e < b->e);
}

int sdm_oracle_plan(int n, int width, const int32_t *slots, int32_t *perm, uint8_t *group_start,
                    uint8_t *owner, uint8_t *only) {
    int m = n * width;
    if (m <= 0) return 0;
    plan_key *keys = (plan_key *)malloc(sizeof(plan_key) * (size_t)m);
    if (!keys) return ORACLE_ENOMEM;
    for (int e = 0; e < m; ++e) { keys[e].slot = slots[e]; keys[e].e = e; }
    qsort(keys, (size_t)m, sizeof(plan_key), plan_cmp);
    int groups = 0;
    for (int i = 0; i < m; ++i) {
        perm[i] = keys[i].e;
        int first = (i == 0) || keys[i].slot != keys[i - 1].slot;
        int last = (i == m - 1) || keys[i].slot != keys[i + 1].slot;
        group_start[i] = (uint8_t)first;
        owner[i] = (uint8_t)last;
        only[i] = (uint8_t)(first && last);
        groups += first;
    }
    free(keys);
    return groups;
}

/* ------------------------------------------------------------------------------------
 * Reverse mode of the token loop, one stream (memory_ops.py: SDMWriteRead.backward's
 * contract: gradients of the readings' loss with respect to the initial bank, v, beta,
 * the write weights, the log-decays and the read weights; the bank is restored to its
 * initial state). Per token, in reverse, with B' the bank after the token and a_j the
 * pre-write rows logged by the forward:
 *   dB'[r_i] += q_i dO ;  dq_i = <dO, B'[r_i]>
 *   dk_j = <dB'[s_j], u> ;  du = sum_j k_j dB'[s_j] ;  dd_j = dB'[s_j]
 *   dbeta = <du, v - ret> ;  dv = beta du ;  dret = -beta du
 *   dk_j += <dret, d_j> ;  dd_j += k_j dret
 *   dg_j = <dd_j, d_j> (= exp(g_j) <dd_j, a_j>) ;  dB[s_j] = exp(g_j) dd_j
 *   restore B[s_j] = a_j
 * ------------------------------------------------------------------------------------ */
/* The reverse pass over tokens t_hi - 1 .. t_lo of one stream (the per-token step above),
 * with B the bank after token t_hi - 1 and a_log the pre-write rows of those tokens; leaves B
 * as it was before token t_lo and adds into dB (the running bank gradient). */
static void reverse_tokens(int t_lo, int t_hi, int D, int W, int R, double *B,
                           const int32_t *ws, const double *k, const double *g,
                           const double *beta, const double *v, const int32_t *rs,
                           const double *q, const double *dout, double *dB, double *dv,
                           double *dbeta, double *dk, double *dg, double *dq,
                           const double *a_log, double *tmp) {
    double *d = tmp;                      /* [W*D] */
    double *dd = d + (size_t)W * D;       /* [W*D] */
    double *du = dd + (size_t)W * D;      /* [D] */
    double *u = du + D;                   /* [D] */
    double *rt = u + D;                   /* [D] */
    for (int t = t_hi - 1; t >= t_lo; --t) {
        const int32_t *s = ws + (size_t)t * W, *r = rs + (size_t)t * R;
        const double *kt = k + (size_t)t * W, *gt = g + (size_t)t * W, *qt = q + (size_t)t * R;
        const double *vt = v + (size_t)t * D, *dO = dout + (size_t)t * D;
        const double *at = a_log + (size_t)t * W * D;
        /* recompute d_j, ret, u of this token from the logged a_j */
        for (int c = 0; c < D; ++c) rt[c] = 0.0;
        for (int j = 0; j < W; ++j) {
            double e = exp(gt[j]);
            for (int c = 0; c < D; ++c) {
                d[(size_t)j * D + c] = e * at[(size_t)j * D + c];
                rt[c] += kt[j] * d[(size_t)j * D + c];
            }
        }
        for (int c = 0; c < D; ++c) u[c] = beta[t] * (vt[c] - rt[c]);
        /* readings */
        for (int i = 0; i < R; ++i) {
            const double *row = B + (size_t)r[i] * D;
            double dot = 0.0;
            for (int c = 0; c < D; ++c) dot += dO[c] * row[c];
            dq[(size_t)t * R + i] = dot;
            double *drow = dB + (size_t)r[i] * D;
            for (int c = 0; c < D; ++c) drow[c] += qt[i] * dO[c];
        }
        /* the write B'[s_j] = d_j + k_j u */
        for (int c = 0; c < D; ++c) du[c] = 0.0;
        for (int j = 0; j < W; ++j) {
            const double *drow = dB + (size_t)s[j] * D;
            double dot = 0.0;
            for (int c = 0; c < D; ++c) {
                dot += drow[c] * u[c];
                du[c] += kt[j] * drow[c];
                dd[(size_t)j * D + c] = drow[c];
            }
            dk[(size_t)t * W + j] = dot;
        }
        /* u = beta (v - ret) */
        double db = 0.0;
        for (int c = 0; c < D; ++c) {
            db += du[c] * (vt[c] - rt[c]);
            dv[(size_t)t * D + c] = beta[t] * du[c];
        }
        dbeta[t] = db;
        /* ret = sum_j k_j d_j (dret = -beta du) ; d_j = exp(g_j) a_j */
        for (int j = 0; j < W; ++j) {
            double dot = 0.0, dgj = 0.0, e = exp(gt[j]);
            for (int c = 0; c < D; ++c) {
                double dret = -beta[t] * du[c];
                dot += dret * d[(size_t)j * D + c];
                dd[(size_t)j * D + c] += kt[j] * dret;
                dgj += dd[(size_t)j * D + c] * d[(size_t)j * D + c];
            }
            dk[(size_t)t * W + j] += dot;
            dg[(size_t)t * W + j] = dgj;
            double *drow = dB + (size_t)s[j] * D;
            double *brow = B + (size_t)s[j] * D;
            for (int c = 0; c < D; ++c) {
                drow[c] = e * dd[(size_t)j * D + c];
                brow[c] = at[(size_t)j * D + c];
            }
        }
    }
}

static int backward_stream(int T, int S, int D, int W, int R, double *B, const int32_t *ws,
                           const double *k, const double *g, const double *beta,
                           const double *v, const int32_t *rs, const double *q, int valid,
                           const double *dout, const double *dB_final, double *dB, double *dv,
                           double *dbeta, double *dk, double *dg, double *dq, double *a_log,
                           double *tmp) {
    double *out = tmp;                    /* [T*D] forward readings (unused) */
    double *a = out + (size_t)T * D;      /* [W*D] */
    double *ret = a + (size_t)W * D;      /* [D] */
    double *rev = ret + D;                /* [2*W*D + 3*D] scratch of reverse_tokens */
    int rc = sequential_stream(T, S, D, W, R, B, ws, k, g, beta, v, rs, q, valid, out, a, ret,
                               a_log);
    if (rc) return rc;
    if (dB_final)
        memcpy(dB, dB_final, sizeof(double) * (size_t)S * D);
    else
        memset(dB, 0, sizeof(double) * (size_t)S * D);
    memset(dv, 0, sizeof(double) * (size_t)T * D);
    memset(dbeta, 0, sizeof(double) * (size_t)T);
    memset(dk, 0, sizeof(double) * (size_t)T * W);
    memset(dg, 0, sizeof(double) * (size_t)T * W);
    memset(dq, 0, sizeof(double) * (size_t)T * R);
    reverse_tokens(0, valid, D, W, R, B, ws, k, g, beta, v, rs, q, dout, dB, dv, dbeta, dk, dg,
                   dq, a_log, rev);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------
 * Reverse mode with a stored snapshot, one stream (memory_ops.py, sdm_write_read docstring:
 * snapshot_quant, "the backward restores ... the written rows to their dequantized snapshot";
 * phase2_kernels.py module docstring: DW stores the snapshot, Phase A restores the rows).
 * The backward walks the chunks in reverse. For chunk c it
 *   1. restores every row the chunk's valid tokens write to Q(its value at the chunk start),
 *      the snapshot the forward kept (Q = identity for "none", bfloat16 rounding for "bf16");
 *   2. re-runs the chunk's tokens from that bank, logging their pre-write rows;
 *   3. takes the reverse pass of those tokens (reverse_tokens), which puts the bank back to
 *      its state at step 1 and carries dB to the chunk before.
 * With Q = identity this is the reverse mode above. For "bf16", Q(x) rounds x first to float32 (the
 * precision of the float32 bank the snapshot is taken from), then to bfloat16, to nearest
 * even: add 0x7fff plus the lowest kept bit to the float32 pattern and clear 16 bits.
 * ------------------------------------------------------------------------------------ */
static double quant_bf16(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Q for "fp8" (memory_ops.py: a snapshot row of head_dim float8_e4m3fn elements, no scale):
 * x rounded to float32, then to the nearest float8_e4m3fn value, ties to the even code, with
 * magnitudes past the largest finite one (448) saturating to it (the format has no infinity;
 * saturation keeps a restored row finite). e4m3fn: exponent bias 7, 3 fraction bits, normal
 * values from 2^-6, subnormal steps of 2^-9. NaN stays NaN. */
static double quant_fp8(double x) {
    double a = (double)(float)x;
    if (a != a) return a;
    const int neg = a < 0;
    a = fabs(a);
    int e;
    frexp(a, &e);                   /* a = f 2^e, 0.5 <= f < 1: the binade's exponent is e - 1 */
    double step = ldexp(1.0, (e - 1 < -6 ? -6 : e - 1) - 3);
    double r = nearbyint(a / step) * step;   /* exact scaling; ties to even (default mode) */
    if (r > 448.0) r = 448.0;
    return neg ? -r : r;
}

static double quant_mode(int mode, double x) {
    return mode == 1 ? quant_bf16(x) : (mode == 2 ? quant_fp8(x) : x);
}

static int backward_snapshot_stream(int T, int C, int S, int D, int W, int R, int mode, double *B,
                                    const int32_t *ws, const double *k, const double *g,
                                    const double *beta, const double *v, const int32_t *rs,
                                    const double *q, int valid, const double *dout,
                                    const double *dB_final, double *dB, double *dv, double *dbeta,
                                    double *dk, double *dg, double *dq, double *a_log,
                                    double *snap, double *tmp) {
    double *out = tmp;                    /* [T*D] readings of the re-runs (unused) */
    double *a = out + (size_t)T * D;      /* [W*D] */
    double *ret = a + (size_t)W * D;      /* [D] */
    double *rev = ret + D;                /* [2*W*D + 3*D] */
    const int Nt = (T + C - 1) / C;
    /* forward, chunk by chunk: the snapshot of each write entry is its row at the chunk start */
    for (int c = 0; c < Nt; ++c) {
        const int t0 = c * C, t1 = t0 + C < valid ? t0 + C : valid;
        for (int t = t0; t < t1; ++t)
            for (int j = 0; j < W; ++j) {
                const int32_t sl = ws[(size_t)t * W + j];
                if (sl < 0 || sl >= S) return ORACLE_EINVAL;
                memcpy(snap + ((size_t)t * W + j) * D, B + (size_t)sl * D, sizeof(double) * D);
            }
        if (t1 > t0) {
            int rc = sequential_stream(t1 - t0, S, D, W, R, B, ws + (size_t)t0 * W,
                                       k + (size_t)t0 * W, g + (size_t)t0 * W, beta + t0,
                                       v + (size_t)t0 * D, rs + (size_t)t0 * R,
                                       q + (size_t)t0 * R, t1 - t0, out, a, ret, NULL);
            if (rc) return rc;
        }
    }
    if (dB_final)
        memcpy(dB, dB_final, sizeof(double) * (size_t)S * D);
    else
        memset(dB, 0, sizeof(double) * (size_t)S * D);
    memset(dv, 0, sizeof(double) * (size_t)T * D);
    memset(dbeta, 0, sizeof(double) * (size_t)T);
    memset(dk, 0, sizeof(double) * (size_t)T * W);
    memset(dg, 0, sizeof(double) * (size_t)T * W);
    memset(dq, 0, sizeof(double) * (size_t)T * R);
    for (int c = Nt - 1; c >= 0; --c) {
        const int t0 = c * C, t1 = t0 + C < valid ? t0 + C : valid;
        if (t1 <= t0) continue;
        /* 1. restore the chunk's written rows from the snapshot */
        for (int t = t0; t < t1; ++t)
            for (int j = 0; j < W; ++j) {
                const double *sr = snap + ((size_t)t * W + j) * D;
                double *row = B + (size_t)ws[(size_t)t * W + j] * D;
                for (int e = 0; e < D; ++e) row[e] = quant_mode(mode, sr[e]);
            }
        /* 2. re-run the chunk, logging the pre-write rows at their tokens */
        int rc = sequential_stream(t1 - t0, S, D, W, R, B, ws + (size_t)t0 * W,
                                   k + (size_t)t0 * W, g + (size_t)t0 * W, beta + t0,
                                   v + (size_t)t0 * D, rs + (size_t)t0 * R, q + (size_t)t0 * R,
                                   t1 - t0, out, a, ret, a_log + (size_t)t0 * W * D);
        if (rc) return rc;
        /* 3. the reverse pass of the chunk's tokens */
        reverse_tokens(t0, t1, D, W, R, B, ws, k, g, beta, v, rs, q, dout, dB, dv, dbeta, dk, dg,
                       dq, a_log, rev);
    }
    return ORACLE_OK;
}

/* Reverse mode with a stored snapshot over all streams (arguments as sdm_oracle_backward,
 * plus the chunk size C and mode 0 = "none", 1 = "bf16", 2 = "fp8"). bank: in = initial bank; out = the
 * bank the backward leaves: every row some valid token writes holds Q(its initial value). */
int sdm_oracle_backward_snapshot(int P, int T, int C, int S, int D, int W, int R, int mode,
                                 double *bank, const int32_t *ws, const double *k,
                                 const double *g, const double *beta, const double *v,
                                 const int32_t *rs, const double *q, const int32_t *valid,
                                 const double *dout, const double *dbank_final, double *dbank,
                                 double *dv, double *dbeta, double *dk, double *dg, double *dq,
                                 int nthreads) {
    if (check_sizes(P, T, S, D, W, R) || C < 1 || mode < 0 || mode > 2) return ORACLE_EINVAL;
    for (int p = 0; p < P; ++p)
        if (valid[p] < 0 || valid[p] > T) return ORACLE_EINVAL;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int p = 0; p < P; ++p) {
        size_t logn = (size_t)T * W * D;
        size_t tmpn = (size_t)T * D + 3 * (size_t)W * D + 4 * (size_t)D;
        double *a_log = (double *)malloc(sizeof(double) * logn);
        double *snap = (double *)malloc(sizeof(double) * logn);
        double *tmp = (double *)malloc(sizeof(double) * tmpn);
        int rc;
        if (!a_log || !snap || !tmp) {
            rc = ORACLE_ENOMEM;
        } else {
            size_t o = (size_t)p * T;
            rc = backward_snapshot_stream(
                T, C, S, D, W, R, mode, bank + (size_t)p * S * D, ws + o * W, k + o * W,
                g + o * W, beta + o, v + o * D, rs + o * R, q + o * R, valid[p], dout + o * D,
                dbank_final ? dbank_final + (size_t)p * S * D : NULL, dbank + (size_t)p * S * D,
                dv + o * D, dbeta + o, dk + o * W, dg + o * W, dq + o * R, a_log, snap, tmp);
        }
        free(a_log);
        free(snap);
        free(tmp);
        if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    return status;
}

/* Forward + reverse over all streams. bank: in = initial bank; out = the initial bank
 * again (the backward restores it exactly). dbank_final (nullable) is the loss gradient with
 * respect to the final bank (zero when NULL). Gradients: dbank [P*S, D] (with respect to the
 * initial bank), dv [P,T,D], dbeta [P,T], dk [P,T,W], dg [P,T,W], dq [P,T,R]. Memory:
 * T*W*D doubles of logged rows per stream in flight. */
int sdm_oracle_backward(int P, int T, int S, int D, int W, int R, double *bank,
                        const int32_t *ws, const double *k, const double *g, const double *beta,
                        const double *v, const int32_t *rs, const double *q,
                        const int32_t *valid, const double *dout, const double *dbank_final,
                        double *dbank, double *dv, double *dbeta, double *dk, double *dg,
                        double *dq, int nthreads) {
    if (check_sizes(P, T, S, D, W, R)) return ORACLE_EINVAL;
    for (int p = 0; p < P; ++p)
        if (valid[p] < 0 || valid[p] > T) return ORACLE_EINVAL;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int p = 0; p < P; ++p) {
        size_t logn = (size_t)T * W * D;
        size_t tmpn = (size_t)T * D + 3 * (size_t)W * D + 4 * (size_t)D;
        double *a_log = (double *)malloc(sizeof(double) * logn);
        double *tmp = (double *)malloc(sizeof(double) * tmpn);
        int rc;
        if (!a_log || !tmp) {
            rc = ORACLE_ENOMEM;
        } else {
            size_t o = (size_t)p * T;
            rc = backward_stream(T, S, D, W, R, bank + (size_t)p * S * D, ws + o * W, k + o * W,
                                 g + o * W, beta + o, v + o * D, rs + o * R, q + o * R,
                                 valid[p], dout + o * D,
                                 dbank_final ? dbank_final + (size_t)p * S * D : NULL,
                                 dbank + (size_t)p * S * D, dv + o * D,
                                 dbeta + o, dk + o * W, dg + o * W, dq + o * R, a_log, tmp);
        }
        free(a_log);
        free(tmp);
        if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    return status;
}
