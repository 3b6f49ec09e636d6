/*
 * fp64 CPU oracle for packed-tree KDA (gated delta rule) forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg load this library.  It shares no code, header or helper with the
 * CUDA library.
 *
 * What it computes.  HARTS (page "HARTS ... 精读", sections 1.1 and 3.2) trains on a
 * rollout tree whose root-to-leaf paths are trajectories; the reference semantics
 * are those of trajectory-wise training.  So this oracle expands the segment tree
 * into its trajectories and runs, per trajectory and head, the recurrence of the
 * KDA layer token by token.  The pages do not print the layer equation ("公式 1");
 * the reading taken is the gated delta rule with per-channel decay,
 *
 *     P_t = diag(exp(g_t)) S_{t-1}
 *     S_t = P_t + beta_t k_t (v_t - P_t^T k_t)^T
 *     o_t = scale * S_t^T q_t,
 *
 * S_0 = 0 (or a given h0 for the tree's root).  The compact output of a row is the
 * output at any of its occurrences (they are the same function of the inputs; the
 * oracle checks they agree).  The backward pass differentiates the loss
 * L = sum_c <W_c, o_c> + <d_final, final states>: W_c is placed on the canonical
 * occurrence of row c (the first trajectory, leaves in increasing segment id,
 * that contains it), the exact token-level reverse sweep runs over every
 * trajectory, and per-occurrence input gradients are summed into compact rows.
 *
 * Reverse sweep for one token (u = v - P^T k):
 *     dS += scale q do^T;    dq = scale S_t do
 *     du = beta dS^T k;      dbeta = k^T dS u;   dv = du
 *     dk = beta dS u - P du
 *     dP = dS - k du^T;      dg_i = sum_j dP_ij P_ij;   dS_{t-1} = diag(exp(g)) dP
 *
 * Memory: states are checkpointed every `ckpt` tokens and recomputed inside a block.
 * Threads: one head per OpenMP thread (heads write disjoint gradient rows).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t n;          /* tokens */
    int64_t *row;       /* compact row per position */
    uint8_t *canon;     /* 1 where this trajectory is the row's canonical occurrence */
    int32_t root;       /* root index */
} traj_t;

static void step_fwd(int dk, int dv, const double *Sprev, const double *kk, const double *vv,
                     const double *gg, double b, double *P, double *u, double *S)
{
    for (int i = 0; i < dk; ++i) {
        double a = exp(gg[i]);
        for (int j = 0; j < dv; ++j) P[i * dv + j] = a * Sprev[i * dv + j];
    }
    for (int j = 0; j < dv; ++j) {
        double s = 0.0;
        for (int i = 0; i < dk; ++i) s += P[i * dv + j] * kk[i];
        u[j] = vv[j] - s;
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[i * dv + j] = P[i * dv + j] + b * kk[i] * u[j];
}

/* Returns 0 on success, -1 on bad input, -2 on allocation failure. */
int oracle_kda_forest(int32_t n_seg, const int32_t *parent, const int64_t *seg_len,
                      const int64_t *seg_off, int32_t H, int32_t dk, int32_t dv,
                      int32_t ckpt, double scale,
                      const double *q, const double *k, const double *v, const double *g,
                      const double *beta, const double *h0, const double *W,
                      const double *d_final, double *o, double *final_state, double *dq,
                      double *dk_out, double *dv_out, double *dg, double *dbeta, double *dh0,
                      int32_t n_threads, double *max_occ_diff)
{
    if (n_seg <= 0 || H <= 0 || dk <= 0 || dv <= 0 || ckpt <= 0) return -1;
    int64_t *start = calloc((size_t)n_seg, sizeof(int64_t));
    int32_t *nkids = calloc((size_t)n_seg, sizeof(int32_t));
    int32_t *canon = malloc((size_t)n_seg * sizeof(int32_t));
    int32_t *rootof = malloc((size_t)n_seg * sizeof(int32_t));
    if (!start || !nkids || !canon || !rootof) return -2;
    int32_t n_roots = 0;
    for (int32_t i = 0; i < n_seg; ++i) {
        int32_t p = parent[i];
        if (p < -1 || p >= i || seg_len[i] < 1) return -1;
        if (p >= 0) { nkids[p]++; start[i] = start[p] + seg_len[p]; rootof[i] = rootof[p]; }
        else { start[i] = 0; rootof[i] = n_roots++; }
    }
    /* canonical leaf of every segment: the smallest leaf id in its subtree */
    for (int32_t i = 0; i < n_seg; ++i) canon[i] = nkids[i] == 0 ? i : INT32_MAX;
    for (int32_t i = n_seg - 1; i >= 0; --i)
        if (parent[i] >= 0 && canon[i] < canon[parent[i]]) canon[parent[i]] = canon[i];

    int32_t n_leaves = 0;
    for (int32_t i = 0; i < n_seg; ++i) n_leaves += nkids[i] == 0;
    traj_t *tr = calloc((size_t)n_leaves, sizeof(traj_t));
    int32_t *path = malloc((size_t)n_seg * sizeof(int32_t));
    if (!tr || !path) return -2;
    int32_t x = 0;
    for (int32_t lf = 0; lf < n_seg; ++lf) {
        if (nkids[lf]) continue;
        int32_t np = 0;
        for (int32_t w = lf; w >= 0; w = parent[w]) path[np++] = w;
        int64_t n = start[lf] + seg_len[lf];
        tr[x].n = n;
        tr[x].root = rootof[lf];
        tr[x].row = malloc((size_t)n * sizeof(int64_t));
        tr[x].canon = malloc((size_t)n);
        if (!tr[x].row || !tr[x].canon) return -2;
        int64_t t = 0;
        for (int32_t a = np - 1; a >= 0; --a) {
            int32_t w = path[a];
            for (int64_t j = 0; j < seg_len[w]; ++j, ++t) {
                tr[x].row[t] = seg_off[w] + j;
                tr[x].canon[t] = canon[w] == lf;
            }
        }
        ++x;
    }
    free(path);

    int64_t C = 0;
    for (int32_t i = 0; i < n_seg; ++i) C += seg_len[i];
    const size_t SS = (size_t)dk * dv;
    if (W) {
        memset(dq, 0, sizeof(double) * (size_t)C * H * dk);
        memset(dk_out, 0, sizeof(double) * (size_t)C * H * dk);
        memset(dv_out, 0, sizeof(double) * (size_t)C * H * dv);
        memset(dg, 0, sizeof(double) * (size_t)C * H * dk);
        memset(dbeta, 0, sizeof(double) * (size_t)C * H);
        if (dh0) memset(dh0, 0, sizeof(double) * (size_t)n_roots * H * SS);
    }
    uint8_t *written = calloc((size_t)C * H, 1);
    if (!written) return -2;
    double occ_diff = 0.0;
    int failed = 0;

#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(max : occ_diff) reduction(| : failed)
#endif
    for (int32_t h = 0; h < H; ++h) {
        int64_t maxn = 0;
        for (int32_t xx = 0; xx < n_leaves; ++xx) if (tr[xx].n > maxn) maxn = tr[xx].n;
        int64_t nck = (maxn + ckpt - 1) / ckpt + 1;
        double *ck = malloc(sizeof(double) * SS * (size_t)nck);
        double *blk = malloc(sizeof(double) * SS * (size_t)(ckpt + 1));
        double *S = malloc(sizeof(double) * SS), *P = malloc(sizeof(double) * SS);
        double *St = malloc(sizeof(double) * SS), *dS = malloc(sizeof(double) * SS);
        double *u = malloc(sizeof(double) * dv), *du = malloc(sizeof(double) * dv);
        if (!ck || !blk || !S || !P || !St || !dS || !u || !du) { failed |= 1; continue; }
        for (int32_t xx = 0; xx < n_leaves; ++xx) {
            const traj_t *T = &tr[xx];
            /* forward with checkpoints: ck[c] = state before token c*ckpt */
            if (h0) memcpy(S, h0 + ((size_t)T->root * H + h) * SS, sizeof(double) * SS);
            else memset(S, 0, sizeof(double) * SS);
            for (int64_t t = 0; t < T->n; ++t) {
                if (t % ckpt == 0) memcpy(ck + SS * (size_t)(t / ckpt), S, sizeof(double) * SS);
                int64_t r = T->row[t];
                const double *kk = k + ((size_t)r * H + h) * dk;
                step_fwd(dk, dv, S, kk, v + ((size_t)r * H + h) * dv, g + ((size_t)r * H + h) * dk,
                         beta[(size_t)r * H + h], P, u, St);
                memcpy(S, St, sizeof(double) * SS);
                const double *qq = q + ((size_t)r * H + h) * dk;
                double *oo = o + ((size_t)r * H + h) * dv;
                uint8_t *wr = &written[(size_t)r * H + h];
                for (int j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < dk; ++i) s += S[i * dv + j] * qq[i];
                    s *= scale;
                    if (!*wr) oo[j] = s;
                    else if (fabs(oo[j] - s) > occ_diff) occ_diff = fabs(oo[j] - s);
                }
                *wr = 1;
            }
            if (final_state) memcpy(final_state + ((size_t)xx * H + h) * SS, S, sizeof(double) * SS);
            if (!W) continue;
            /* reverse sweep */
            if (d_final) memcpy(dS, d_final + ((size_t)xx * H + h) * SS, sizeof(double) * SS);
            else memset(dS, 0, sizeof(double) * SS);
            int64_t nb = (T->n + ckpt - 1) / ckpt;
            for (int64_t bi = nb - 1; bi >= 0; --bi) {
                int64_t t0 = bi * ckpt, t1 = t0 + ckpt < T->n ? t0 + ckpt : T->n;
                memcpy(blk, ck + SS * (size_t)bi, sizeof(double) * SS);   /* blk[j] = S_{t0+j-1} */
                for (int64_t t = t0; t < t1 - 1; ++t) {
                    int64_t r = T->row[t];
                    step_fwd(dk, dv, blk + SS * (size_t)(t - t0), k + ((size_t)r * H + h) * dk,
                             v + ((size_t)r * H + h) * dv, g + ((size_t)r * H + h) * dk,
                             beta[(size_t)r * H + h], P, u, blk + SS * (size_t)(t - t0 + 1));
                }
                for (int64_t t = t1 - 1; t >= t0; --t) {
                    int64_t r = T->row[t];
                    size_t rh = (size_t)r * H + h;
                    const double *kk = k + rh * dk, *gg = g + rh * dk, *qq = q + rh * dk;
                    double b = beta[rh];
                    step_fwd(dk, dv, blk + SS * (size_t)(t - t0), kk, v + rh * dv, gg, b, P, u, St);
                    if (T->canon[t]) {
                        const double *dO = W + rh * dv;
                        for (int i = 0; i < dk; ++i) {
                            double s = 0.0;
                            for (int j = 0; j < dv; ++j) s += St[i * dv + j] * dO[j];
                            dq[rh * dk + i] += scale * s;
                            for (int j = 0; j < dv; ++j) dS[i * dv + j] += scale * qq[i] * dO[j];
                        }
                    }
                    double db = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        double s = 0.0;
                        for (int i = 0; i < dk; ++i) s += kk[i] * dS[i * dv + j];
                        du[j] = b * s;
                        db += s * u[j];
                    }
                    dbeta[rh] += db;
                    for (int j = 0; j < dv; ++j) dv_out[rh * dv + j] += du[j];
                    for (int i = 0; i < dk; ++i) {
                        double s1 = 0.0, s2 = 0.0;
                        for (int j = 0; j < dv; ++j) { s1 += dS[i * dv + j] * u[j]; s2 += P[i * dv + j] * du[j]; }
                        dk_out[rh * dk + i] += b * s1 - s2;
                    }
                    for (int i = 0; i < dk; ++i) {
                        double a = exp(gg[i]), s = 0.0;
                        for (int j = 0; j < dv; ++j) {
                            double dp = dS[i * dv + j] - kk[i] * du[j];
                            s += dp * P[i * dv + j];
                            dS[i * dv + j] = a * dp;
                        }
                        dg[rh * dk + i] += s;
                    }
                }
            }
            if (dh0) {
                double *d = dh0 + ((size_t)T->root * H + h) * SS;
                for (size_t e = 0; e < SS; ++e) d[e] += dS[e];
            }
        }
        free(ck); free(blk); free(S); free(P); free(St); free(dS); free(u); free(du);
    }
    for (int32_t xx = 0; xx < n_leaves; ++xx) { free(tr[xx].row); free(tr[xx].canon); }
    free(tr); free(start); free(nkids); free(canon); free(rootof); free(written);
    if (max_occ_diff) *max_occ_diff = occ_diff;
    return failed ? -2 : 0;
}
